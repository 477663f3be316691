import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library (fails loudly if it is missing)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_qk_norm_gb300 import binding
    return binding.load()
