"""K1 (QK-Norm + RoPE) on the GPU against the fp64 oracle, through the C ABI."""
import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import binding, inputs
from gpu_util import assert_within_one_ulp

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,T,H,pos0,theta", [
    (1, 5, 3, 0, 1e6), (2, 37, 8, 0, 1e6), (1, 9, 32, 32759, 1e6), (3, 2, 4, 0, 1e7),
    (1, 4, 2, (1 << 30) - 3, 1e7), (1, 131, 1, 7, 1e4)])
def test_qknorm_rope_matches_oracle(cuda_lib, B, T, H, pos0, theta):
    x = inputs.prefill_inputs(B, T, H, H, seed=100 + T, outlier_frac=0.1, outlier_scale=30.0)
    ref = oracle.qknorm_rope(x["q"], x["q_gamma"], theta, 1e-6, pos0=pos0)
    got = binding.qknorm_rope(x["q"].cuda(), x["q_gamma"].cuda(), theta, 1e-6, pos0=pos0)
    torch.cuda.synchronize()
    assert_within_one_ulp(got, ref, "qknorm_rope")


def test_qknorm_rope_in_place(cuda_lib):
    x = inputs.prefill_inputs(2, 17, 5, 5, seed=7)
    ref = oracle.qknorm_rope(x["q"], x["q_gamma"], 1e6, 1e-6)
    xd = x["q"].cuda()
    binding.qknorm_rope(xd, x["q_gamma"].cuda(), 1e6, 1e-6, out=xd)
    torch.cuda.synchronize()
    assert_within_one_ulp(xd, ref, "in place")


def test_qknorm_rope_zero_rows_stay_zero(cuda_lib):
    x = torch.zeros((1, 3, 2, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(128, dtype=torch.bfloat16, device="cuda")
    y = binding.qknorm_rope(x, g, 1e6, 1e-6, pos0=11)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y) == 0
