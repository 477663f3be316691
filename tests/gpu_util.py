"""Helpers shared by the GPU parity tests (comparison and tolerance)."""
import torch

# Tolerance of the attention outputs against the fp64 oracle: bf16 outputs,
# max-abs <= 2e-2 and mean-abs <= 2e-3.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def assert_close_attention(got_bf16: torch.Tensor, ref_f64: torch.Tensor, what: str = ""):
    got = got_bf16.detach().to("cpu", torch.float64)
    ref = ref_f64.to(torch.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert torch.isfinite(got).all(), f"{what}: non-finite output"
    err = (got - ref).abs()
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max-abs {mx:.3e} mean-abs {mean:.3e}"
    return mx, mean


def bf16_ulp(x: torch.Tensor) -> torch.Tensor:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = x.abs().clamp_min(2.0 ** -126)
    return torch.exp2(torch.floor(torch.log2(ax)) - 7)


def assert_within_one_ulp(got_bf16: torch.Tensor, ref_f64: torch.Tensor, what: str = ""):
    """A once-rounded fp32 result against the exact value: at most one bf16 ulp."""
    got = got_bf16.detach().to("cpu", torch.float64)
    ref = ref_f64.to(torch.float64)
    err = (got - ref).abs()
    bound = bf16_ulp(ref) + 1e-6
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off by more than 1 ulp, worst {float((err - bound).max()):.3e}"
