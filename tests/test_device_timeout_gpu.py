"""The device-side timeout path: a bounded mbarrier wait that runs out records
its code in the error word, the kernel returns (no trap, no hang), the host
reads Q3A_ETIMEOUT, and the context stays usable for the next call (the clear
errors of "Chapter 20, Qwen3 and Qwen3.5" §20.9)."""
import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import binding, inputs
from gpu_util import assert_close_attention

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_etimeout_and_context_stays_usable(cuda_lib):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    # nothing arrives: the wait gives up after about 0.1 ms of SM cycles
    binding.selftest_bounded_wait(ws, limit_cycles=200_000, arrive=False)
    torch.cuda.synchronize()
    assert binding.last_device_error(ws) == binding.Q3A_ETIMEOUT
    assert int(ws[:4].view(torch.int32).item()) == 0x106
    # the barrier completes: the word is cleared and stays zero
    binding.selftest_bounded_wait(ws, limit_cycles=200_000, arrive=True)
    assert binding.last_device_error(ws) == binding.Q3A_OK
    # the same context still computes correctly
    x = inputs.prefill_inputs(1, 130, 8, 2, seed=61)
    d = {k: t.cuda() for k, t in x.items()}
    out = binding.prefill(d["q"], d["k"], d["v"], d["q_gamma"], d["k_gamma"], 1e6, 1e-6)
    torch.cuda.synchronize()
    ref = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    assert_close_attention(out, ref, "prefill after a device timeout")


def test_selftest_rejects_bad_arguments(cuda_lib):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.Q3AError) as e:
        binding.selftest_bounded_wait(ws, limit_cycles=0, arrive=False)
    assert e.value.status == binding.Q3A_EINVAL
    with pytest.raises(binding.Q3AError) as e:
        binding.selftest_bounded_wait(ws[:128], limit_cycles=1000, arrive=False)
    assert e.value.status == binding.Q3A_EINVAL
