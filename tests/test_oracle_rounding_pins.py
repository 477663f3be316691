"""Pins of the oracle's bf16-rounded prefill (``oracle.prefill_rounded``), the
reference for large gammas.

"7.2 Qwen3 full-scale implementation" §7.2.1 casts the normalised rows back to
the model dtype (RMSNorm returns ``.to(input_dtype)``) and the rotated rows too
(``apply_rope`` returns ``.to(dtype=x.dtype)``): a bf16 model multiplies bf16
q-hat and k-hat. With large gammas the logits are large and those roundings
alone move the attention output by more than the bf16 output tolerance, so the
fp64 oracle without roundings cannot judge a bf16 implementation there. These
tests fix the rounding itself (nearest bf16, ties to even), pin the rounded
prefill to a separately written brute force, and record, as executable claims,
how far the roundings alone move the output at each gamma.
"""
import math

import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import inputs

D = 128
HALF = D // 2


def _py_round_bf16(x: float) -> float:
    """Nearest bf16 value (8 significant bits), ties to even: Python's round()
    on the value scaled to an integer spacing (normal range only)."""
    if x == 0.0:
        return x
    _, e = math.frexp(x)
    return math.ldexp(round(math.ldexp(x, 8 - e)), e - 8)


def _bf16_neighbours(r: torch.Tensor):
    """The bf16 values just below and above each (positive, normal) r."""
    bits = r.to(torch.bfloat16).view(torch.int16)
    down = (bits - 1).view(torch.bfloat16).to(torch.float64)
    up = (bits + 1).view(torch.bfloat16).to(torch.float64)
    return down, up


def test_round_bf16_matches_torch_on_fp32_values():
    """On fp32 inputs, including exact ties (low 16 bits 0x8000, both parities),
    the oracle's rounding equals torch's fp32 -> bf16 conversion."""
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(0, 2 ** 31 - 1, (20000,), generator=g, dtype=torch.int64)
    bits = bits[((bits >> 23) & 0xFF) < 0xFE]  # finite, below the bf16 overflow edge
    ties = (bits & ~0xFFFF) | 0x8000
    allb = torch.cat([bits, ties]).to(torch.int32)
    f32 = allb.view(torch.float32)
    f32 = torch.cat([f32, -f32])
    want = f32.to(torch.bfloat16).to(torch.float64)
    got = oracle.round_bf16(f32.to(torch.float64))
    assert torch.equal(got, want)


def test_round_bf16_is_nearest_with_ties_to_even():
    g = torch.Generator().manual_seed(4)
    x = torch.exp(torch.randn(20000, generator=g, dtype=torch.float64) * 15)  # about 1e-29 .. 1e29
    r = oracle.round_bf16(x)
    down, up = _bf16_neighbours(r)
    assert torch.equal(r.to(torch.bfloat16).to(torch.float64), r)  # a bf16 value
    assert bool(((x - r).abs() <= (x - down).abs()).all())
    assert bool(((x - r).abs() <= (x - up).abs()).all())
    # exact midpoints between two bf16 values go to the one with an even mantissa
    lo = torch.tensor([1.0, 1.0078125, 3.0, 1000.0, 2.0 ** -100]).to(torch.bfloat16)
    hi = (lo.view(torch.int16) + 1).view(torch.bfloat16)
    mid = (lo.double() + hi.double()) / 2
    got = oracle.round_bf16(mid)
    even = torch.where(lo.view(torch.int16) % 2 == 0, lo.double(), hi.double())
    assert torch.equal(got, even)
    assert torch.equal(oracle.round_bf16(-mid), -even)


def test_round_bf16_of_the_python_rounding():
    """The brute force below uses a separately written rounding; both agree."""
    g = torch.Generator().manual_seed(5)
    x = torch.randn(5000, generator=g, dtype=torch.float64) * 7
    got = oracle.round_bf16(x).tolist()
    assert got == [_py_round_bf16(v) for v in x.tolist()]


def _brute_force_rounded(x, theta, eps, roundings):
    """Separately written: per-row norm with math.fsum, explicit 2x2 rotation
    blocks, the Python rounding after the norm (roundings == 2) and after the
    rotation (roundings >= 1), a softmax without max subtraction."""
    q, k, v = (x[n].to(torch.float64).tolist() for n in ("q", "k", "v"))
    gq = x["q_gamma"].to(torch.float64).tolist()
    gk = x["k_gamma"].to(torch.float64).tolist()
    B, T, Hq = len(q), len(q[0]), len(q[0][0])
    Hkv = len(k[0][0])
    g = Hq // Hkv

    def prep(row, gamma, p):
        inv = 1.0 / math.sqrt(math.fsum(e * e for e in row) / D + eps)
        y = [row[c] * inv * gamma[c] for c in range(D)]
        if roundings == 2:
            y = [_py_round_bf16(e) for e in y]
        res = [0.0] * D
        for i in range(HALF):
            ang = p * theta ** (-2.0 * i / D)
            c, s = math.cos(ang), math.sin(ang)
            res[i] = c * y[i] - s * y[i + HALF]
            res[i + HALF] = s * y[i] + c * y[i + HALF]
        if roundings >= 1:
            res = [_py_round_bf16(e) for e in res]
        return res

    out = torch.zeros((B, T, Hq, D), dtype=torch.float64)
    for b in range(B):
        khat = [[prep(k[b][j][kv], gk, j) for kv in range(Hkv)] for j in range(T)]
        for i in range(T):
            for h in range(Hq):
                grp = h // g
                qh = prep(q[b][i][h], gq, i)
                w = [math.exp(math.fsum(qh[c] * khat[j][grp][c] for c in range(D)) / math.sqrt(D))
                     for j in range(i + 1)]
                z = math.fsum(w)
                for c in range(D):
                    out[b, i, h, c] = math.fsum(w[j] * v[b][j][grp][c] for j in range(i + 1)) / z
    return out


def test_prefill_rounded_without_roundings_is_prefill():
    x = inputs.prefill_inputs(2, 40, 8, 2, seed=21)
    a = [x[n] for n in ("q", "k", "v", "q_gamma", "k_gamma")]
    assert torch.equal(oracle.prefill_rounded(*a, 1e6, 1e-6, 0), oracle.prefill(*a, 1e6, 1e-6))


@pytest.mark.parametrize("roundings", [1, 2])
@pytest.mark.parametrize("B,T,Hq,Hkv,theta,seed", [(1, 7, 2, 1, 1e6, 22), (2, 5, 4, 2, 1e4, 23)])
def test_prefill_rounded_matches_brute_force(B, T, Hq, Hkv, theta, seed, roundings):
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=seed)
    g = torch.Generator().manual_seed(seed)
    x["q_gamma"] = (torch.rand(D, generator=g) * 4).to(torch.bfloat16)  # large logits
    a = [x[n] for n in ("q", "k", "v", "q_gamma", "k_gamma")]
    got = oracle.prefill_rounded(*a, theta, 1e-6, roundings)
    ref = _brute_force_rounded(x, theta, 1e-6, roundings)
    assert (got - ref).abs().max() < 1e-12
    # the roundings do act: the result differs from the unrounded prefill
    assert (got - oracle.prefill(*a, theta, 1e-6)).abs().max() > 1e-6


def _gamma_case(gmax):
    """The 300-token case of the GPU softmax-path tests: gammas ~ U(0, gmax)."""
    x = inputs.prefill_inputs(1, 300, 16, 4, seed=int(gmax * 10))
    g = torch.Generator().manual_seed(77)
    x["q_gamma"] = (torch.rand(D, generator=g) * gmax).to(torch.bfloat16)
    x["k_gamma"] = (torch.rand(D, generator=g) * gmax).to(torch.bfloat16)
    return [x[n] for n in ("q", "k", "v", "q_gamma", "k_gamma")]


@pytest.mark.parametrize("gmax,lo,hi", [(1.5, 3e-3, 6e-3), (2.3, 1.5e-2, 1.9e-2),
                                        (2.5, 2.2e-2, 2.8e-2), (6.0, 1.0e-1, 1.6e-1)])
def test_bf16_qhat_khat_alone_move_the_output_with_gamma(gmax, lo, hi):
    """Max-abs distance between the exact fp64 output and the one computed from
    bf16-rounded qhat and khat (nothing else rounded): it grows with the logit
    scale sqrt(128) max|gamma_q| max|gamma_k|, from 4.8e-3 at gamma <= 1.5 to
    past the 2e-2 output tolerance at gamma <= 2.5 (2.5e-2) and 6 (0.13). A bf16
    kernel, whose attention products take bf16 operands, is therefore compared
    with the exact oracle only up to gamma 2.3 and with the rounded one above."""
    a = _gamma_case(gmax)
    exact = oracle.prefill(*a, 1e6, 1e-6)
    r1 = oracle.prefill_rounded(*a, 1e6, 1e-6, 1)
    mx = float((r1 - exact).abs().max())
    assert lo < mx < hi, mx


def test_the_pages_double_rounding_moves_it_further():
    """The pages' own bf16 model rounds twice (after the norm and after RoPE);
    at gamma <= 2.5 that alone is 3.2e-2 from the exact output, and 3.9e-2
    from the once-rounded one."""
    a = _gamma_case(2.5)
    exact = oracle.prefill(*a, 1e6, 1e-6)
    r1 = oracle.prefill_rounded(*a, 1e6, 1e-6, 1)
    r2 = oracle.prefill_rounded(*a, 1e6, 1e-6, 2)
    assert 2.9e-2 < float((r2 - exact).abs().max()) < 3.5e-2
    assert 3.5e-2 < float((r2 - r1).abs().max()) < 4.2e-2
