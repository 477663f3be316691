"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against a closed form, an invariant of the
mathematics, a value the pages print, or a separately written brute force, so
that a plausible slip in the oracle (a dropped term, a wrong sign, a wrong
pairing or index, eps outside the square root, the wrong GQA map, an off-by-one
in the causal mask) fails at least one of them.
"""
import json
import math
import os

import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import inputs
from qwen3_qk_norm_gb300.accounting import kv_cache_bytes_per_token

D = 128
HALF = D // 2
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_randn(*shape, seed=0, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def widened(t):
    return [float(x) for x in t.to(torch.float64).flatten()]


# ----------------------------------------------------------------------------
# Step 1: RMSNorm (§7.2.1 RMSNorm; the Qwen1->3 blog's RMS(x) = sqrt(eps + mean x^2))
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("eps", [1e-6, 1.0, 4.0])
def test_rmsnorm_unit_gamma_has_closed_form_rms(eps):
    """With gamma = 1 the output RMS is sqrt(ms / (ms + eps)): eps sits inside the root."""
    ones = torch.ones(D, dtype=torch.bfloat16)
    for seed in range(4):
        x = bf16_randn(D, seed=seed)
        y = oracle.rmsnorm_row(x, ones, eps)
        ms = math.fsum(v * v for v in widened(x)) / D
        rms_y = math.sqrt(math.fsum(v * v for v in y.tolist()) / D)
        assert rms_y == pytest.approx(math.sqrt(ms / (ms + eps)), rel=1e-13)


def test_rmsnorm_gamma_is_elementwise_per_dim():
    x = bf16_randn(D, seed=1)
    gamma = (torch.rand(D, generator=torch.Generator().manual_seed(2)) + 0.5).to(torch.bfloat16)
    y1 = oracle.rmsnorm_row(x, torch.ones(D, dtype=torch.bfloat16), 1e-6)
    yg = oracle.rmsnorm_row(x, gamma, 1e-6)
    assert torch.allclose(yg, y1 * gamma.to(torch.float64), rtol=1e-15, atol=0)


def test_rmsnorm_direction_preserved_and_scale_invariant():
    """RMSNorm(c x) = RMSNorm(x) up to the eps term; exact powers of two keep bf16 exact."""
    x = bf16_randn(D, seed=3)
    gamma = torch.ones(D, dtype=torch.bfloat16)
    y = oracle.rmsnorm_row(x, gamma, 1e-6)
    y32 = oracle.rmsnorm_row((x.to(torch.float32) * 32).to(torch.bfloat16), gamma, 1e-6)
    assert torch.allclose(y, y32, rtol=1e-6, atol=0)
    # the x30 norm outliers of the 8B workload: equal to bf16 rounding of 30x
    y30 = oracle.rmsnorm_row((x.to(torch.float32) * 30).to(torch.bfloat16), gamma, 1e-6)
    assert (y - y30).abs().max() < 2e-2
    # output is parallel to the input
    xd = x.to(torch.float64)
    cos = torch.dot(xd, y) / (xd.norm() * y.norm())
    assert cos == pytest.approx(1.0, abs=1e-14)


def test_rmsnorm_zero_row_is_zero():
    z = torch.zeros(D, dtype=torch.bfloat16)
    y = oracle.rmsnorm_row(z, torch.ones(D, dtype=torch.bfloat16), 1e-6)
    assert torch.count_nonzero(y) == 0


# ----------------------------------------------------------------------------
# Step 2: rotate-half RoPE (§7.2.1 compute_rope_params / apply_rope)
# ----------------------------------------------------------------------------

def basis(i):
    e = torch.zeros(D, dtype=torch.float64)
    e[i] = 1.0
    return e


def test_rope_position_zero_is_identity():
    y = torch.randn(D, dtype=torch.float64, generator=torch.Generator().manual_seed(4))
    assert torch.equal(oracle.rope_row(y, 0, 1e6), y)


@pytest.mark.parametrize("i,pos,theta", [(0, 1, 1e6), (32, 1000, 1e6), (32, 100, 1e4),
                                         (0, 1, 1e7), (16, 10, 1e4)])
def test_rope_exact_angles_of_basis_vectors(i, pos, theta):
    """e_i (i < d/2) -> cos(a) e_i + sin(a) e_{i+d/2}; e_{i+d/2} -> -sin(a) e_i + cos(a) e_{i+d/2}.

    Angles chosen so that pos * theta^(-2i/d) is a round number: i=0, p=1 is
    1 rad for every theta; i=32 is theta^(-1/2) (1e-3 for 1e6, 1e-2 for 1e4);
    i=16, theta=1e4 is 10^-1, so p=10 is 1 rad. A wrong exponent (i/d instead
    of 2i/d), a swapped sign or interleaved pairs fail here.
    """
    a = {(0, 1): 1.0, (32, 1000): 1.0, (32, 100): 1.0, (16, 10): 1.0}[(i, pos)]
    lo = oracle.rope_row(basis(i), pos, theta)
    hi = oracle.rope_row(basis(i + HALF), pos, theta)
    exp_lo = torch.zeros(D, dtype=torch.float64)
    exp_lo[i], exp_lo[i + HALF] = math.cos(a), math.sin(a)
    exp_hi = torch.zeros(D, dtype=torch.float64)
    exp_hi[i], exp_hi[i + HALF] = -math.sin(a), math.cos(a)
    assert torch.allclose(lo, exp_lo, atol=1e-12, rtol=0)
    assert torch.allclose(hi, exp_hi, atol=1e-12, rtol=0)


def test_rope_preserves_pair_norms():
    y = torch.randn(D, dtype=torch.float64, generator=torch.Generator().manual_seed(5))
    for pos in [1, 17, 4095, 32767]:
        r = oracle.rope_row(y, pos, 1e6)
        n0 = y[:HALF] ** 2 + y[HALF:] ** 2
        n1 = r[:HALF] ** 2 + r[HALF:] ** 2
        assert torch.allclose(n0, n1, rtol=1e-13, atol=0)


@pytest.mark.parametrize("delta", [1, 1000, 30000])
def test_rope_scores_depend_only_on_relative_position(delta):
    g = torch.Generator().manual_seed(6)
    q = torch.randn(D, dtype=torch.float64, generator=g)
    k = torch.randn(D, dtype=torch.float64, generator=g)
    for m, n in [(0, 5), (7, 3), (100, 2000)]:
        s0 = torch.dot(oracle.rope_row(q, m, 1e6), oracle.rope_row(k, n, 1e6))
        s1 = torch.dot(oracle.rope_row(q, m + delta, 1e6), oracle.rope_row(k, n + delta, 1e6))
        assert float(s0) == pytest.approx(float(s1), abs=1e-9)


def test_rope_rotations_compose():
    y = torch.randn(D, dtype=torch.float64, generator=torch.Generator().manual_seed(7))
    two = oracle.rope_row(oracle.rope_row(y, 300, 1e6), 700, 1e6)
    one = oracle.rope_row(y, 1000, 1e6)
    assert torch.allclose(two, one, atol=1e-11, rtol=0)


def test_qknorm_rope_is_norm_then_rope():
    """The reading taken where the pages disagree: RMSNorm first, then RoPE.

    With a non-uniform gamma the two orders give different results, so this
    test would catch a swap.
    """
    x = bf16_randn(1, 3, 2, D, seed=8)
    gamma = (torch.rand(D, generator=torch.Generator().manual_seed(9)) + 0.5).to(torch.bfloat16)
    y = oracle.qknorm_rope(x, gamma, 1e6, 1e-6, pos0=5)
    for t in range(3):
        for h in range(2):
            ref = oracle.rope_row(oracle.rmsnorm_row(x[0, t, h], gamma, 1e-6), 5 + t, 1e6)
            assert torch.equal(y[0, t, h], ref)
    # the other order differs (gamma does not commute with the rotation)
    xr = oracle.rope_row(x[0, 2, 0].to(torch.float64), 7, 1e6)
    ms = float((xr ** 2).mean())
    other = xr / math.sqrt(ms + 1e-6) * gamma.to(torch.float64)
    assert (other - y[0, 2, 0]).abs().max() > 1e-2


# ----------------------------------------------------------------------------
# Steps 3-5: GQA map, causal mask, softmax attention
# ----------------------------------------------------------------------------

def test_prefill_row0_equals_v_row0_of_its_group():
    B, T, Hq, Hkv = 2, 9, 8, 2
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=10)
    out = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            assert torch.allclose(out[b, 0, h], x["v"][b, 0, h // g].to(torch.float64),
                                  atol=1e-15, rtol=0)


def test_zero_queries_average_the_causal_prefix():
    """q = 0 normalises to 0, all scores are 0, softmax is uniform over j <= i."""
    B, T, Hq, Hkv = 1, 7, 4, 2
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=11)
    q = torch.zeros_like(x["q"])
    out = oracle.prefill(q, x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    v = x["v"].to(torch.float64)
    for i in range(T):
        for h in range(Hq):
            ref = v[0, : i + 1, h // 2].mean(dim=0)
            assert torch.allclose(out[0, i, h], ref, atol=1e-14, rtol=0)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (8, 2), (16, 2), (16, 1)])
def test_gqa_head_to_group_map_matches_both_page_formulas(Hq, Hkv):
    """The blog's 1-based map u = floor((t-1)/g) + 1 and §7.2.1's repeat_interleave."""
    T, g = 3, Hq // Hkv
    q = torch.zeros((1, T, Hq, D), dtype=torch.bfloat16)
    k = bf16_randn(1, T, Hkv, D, seed=12)
    v = torch.empty((1, T, Hkv, D), dtype=torch.bfloat16)
    for kv in range(Hkv):
        v[:, :, kv, :] = float(kv + 1)          # value rows identify their group
    ones = torch.ones(D, dtype=torch.bfloat16)
    out = oracle.prefill(q, k, v, ones, ones, 1e6, 1e-6)
    group_of_head = torch.repeat_interleave(torch.arange(Hkv), g)
    for h in range(Hq):
        t1 = h + 1                                # 1-based head index
        u = (t1 - 1) // g + 1                     # 1-based group index
        assert float(out[0, T - 1, h, 0]) == pytest.approx(u)
        assert u - 1 == int(group_of_head[h])


def _brute_force_prefill(x, theta, eps):
    """Separately written brute force: explicit 2x2 rotation blocks, a
    softmax without max subtraction, the 1-based GQA map and math-module sums.
    Tiny inputs only."""
    q, k, v = (x[n].to(torch.float64).tolist() for n in ("q", "k", "v"))
    gq = x["q_gamma"].to(torch.float64).tolist()
    gk = x["k_gamma"].to(torch.float64).tolist()
    B, T, Hq = len(q), len(q[0]), len(q[0][0])
    Hkv = len(k[0][0])
    g = Hq // Hkv

    def norm(row, gamma):
        inv = 1.0 / math.sqrt(math.fsum(e * e for e in row) / D + eps)
        return [row[c] * inv * gamma[c] for c in range(D)]

    def rotate(row, p):
        res = [0.0] * D
        for i in range(HALF):
            ang = p * theta ** (-2.0 * i / D)
            c, s = math.cos(ang), math.sin(ang)
            # [[c, -s], [s, c]] acting on the pair (row[i], row[i + HALF])
            res[i] = c * row[i] - s * row[i + HALF]
            res[i + HALF] = s * row[i] + c * row[i + HALF]
        return res

    out = torch.zeros((B, T, Hq, D), dtype=torch.float64)
    for b in range(B):
        khat = [[rotate(norm(k[b][j][kv], gk), j) for kv in range(Hkv)] for j in range(T)]
        for i in range(T):
            for h in range(Hq):
                grp = ((h + 1) - 1) // g + 1 - 1
                qh = rotate(norm(q[b][i][h], gq), i)
                w = [math.exp(math.fsum(qh[c] * khat[j][grp][c] for c in range(D))
                              / math.sqrt(D)) for j in range(i + 1)]
                z = math.fsum(w)
                for c in range(D):
                    out[b, i, h, c] = math.fsum(w[j] * v[b][j][grp][c] for j in range(i + 1)) / z
    return out


@pytest.mark.parametrize("B,T,Hq,Hkv,theta,seed", [(1, 6, 2, 1, 1e6, 13), (2, 5, 4, 2, 1e7, 14),
                                                   (1, 9, 4, 4, 1e4, 15)])
def test_prefill_matches_brute_force(B, T, Hq, Hkv, theta, seed):
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=seed)
    got = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], theta, 1e-6)
    ref = _brute_force_prefill(x, theta, 1e-6)
    assert (got - ref).abs().max() < 1e-12


def test_prefill_rows_equal_full_prefill():
    B, T, Hq, Hkv = 2, 33, 8, 2
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=16, outlier_frac=0.1, outlier_scale=30.0)
    full = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    rows = torch.tensor([[0, 0, 0], [1, 32, 7], [0, 17, 3], [1, 5, 4]], dtype=torch.int32)
    part = oracle.prefill_rows(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6,
                               rows)
    for s, (b, t, h) in enumerate(rows.tolist()):
        assert torch.allclose(part[s], full[b, t, h], atol=1e-14, rtol=0)


def test_future_tokens_do_not_change_past_rows():
    """Causality (the 'future-token invariance' check of §20.8): changing keys
    and values after row i leaves rows 0..i unchanged, exactly."""
    B, T, Hq, Hkv, cut = 1, 12, 4, 2, 6
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=17)
    y = dict(x)
    y["k"] = x["k"].clone()
    y["v"] = x["v"].clone()
    y["k"][:, cut:] = bf16_randn(B, T - cut, Hkv, D, seed=18)
    y["v"][:, cut:] = bf16_randn(B, T - cut, Hkv, D, seed=19)
    a = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    b = oracle.prefill(y["q"], y["k"], y["v"], y["q_gamma"], y["k_gamma"], 1e6, 1e-6)
    assert torch.equal(a[:, :cut], b[:, :cut])
    assert not torch.equal(a[:, cut:], b[:, cut:])


def test_outlier_rows_are_tamed_by_the_norm():
    """Scaling a Q row by an exact power of two leaves its attention output unchanged."""
    B, T, Hq, Hkv = 1, 10, 2, 1
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=20)
    a = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    q2 = (x["q"].to(torch.float32) * 32).to(torch.bfloat16)
    k2 = (x["k"].to(torch.float32) * 32).to(torch.bfloat16)
    b = oracle.prefill(q2, k2, x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    # only the eps term moves: relative change of each normalised row is about
    # eps / (2 ms) = 5e-7, scores are O(10), so outputs move by O(1e-5)
    assert (a - b).abs().max() < 5e-5
    # and a dropped norm would move them by O(1)
    assert (a - b).abs().max() > 0


# ----------------------------------------------------------------------------
# Decode (§20.3: rotate the new key at start_pos, keep cached keys as stored)
# ----------------------------------------------------------------------------

def test_decode_at_position_zero_returns_v_new():
    B, Hq, Hkv, S = 3, 8, 2, 4
    x = inputs.decode_inputs(B, Hq, Hkv, S, 0, 1, seed=21, start_pos=[0, 0, 0])
    out, k_row = oracle.decode(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                               x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    for b in range(B):
        for h in range(Hq):
            assert torch.allclose(out[b, h], x["v_new"][b, h // 4].to(torch.float64),
                                  atol=1e-15, rtol=0)
        for kv in range(Hkv):   # RoPE at position 0 is the identity
            ref = oracle.rmsnorm_row(x["k_new"][b, kv], x["k_gamma"], 1e-6)
            assert torch.allclose(k_row[b, kv], ref, atol=0, rtol=0)


def _brute_force_decode(x, theta, eps):
    q, kn, vn = (x[n].to(torch.float64).tolist() for n in ("q", "k_new", "v_new"))
    kc, vc = x["k_cache"].to(torch.float64), x["v_cache"].to(torch.float64)
    gq = x["q_gamma"].to(torch.float64).tolist()
    gk = x["k_gamma"].to(torch.float64).tolist()
    B, Hq, Hkv = len(q), len(q[0]), len(kn[0])
    g = Hq // Hkv

    def norm(row, gamma):
        inv = 1.0 / math.sqrt(math.fsum(e * e for e in row) / D + eps)
        return [row[c] * inv * gamma[c] for c in range(D)]

    def rotate(row, p):
        res = [0.0] * D
        for i in range(HALF):
            ang = p * theta ** (-2.0 * i / D)
            c, s = math.cos(ang), math.sin(ang)
            res[i] = c * row[i] - s * row[i + HALF]
            res[i + HALF] = s * row[i] + c * row[i + HALF]
        return res

    out = torch.zeros((B, Hq, D), dtype=torch.float64)
    for b in range(B):
        p = int(x["start_pos"][b])
        for h in range(Hq):
            kv = h // g
            keys = [kc[b, kv, j].tolist() for j in range(p)] + [rotate(norm(kn[b][kv], gk), p)]
            vals = [vc[b, kv, j].tolist() for j in range(p)] + [vn[b][kv]]
            qh = rotate(norm(q[b][h], gq), p)
            w = [math.exp(math.fsum(qh[c] * kr[c] for c in range(D)) / math.sqrt(D)) for kr in keys]
            z = math.fsum(w)
            for c in range(D):
                out[b, h, c] = math.fsum(w[j] * vals[j][c] for j in range(len(keys))) / z
    return out


def test_decode_matches_brute_force_with_cache_used_as_stored():
    B, Hq, Hkv, S = 2, 4, 2, 12
    x = inputs.decode_inputs(B, Hq, Hkv, S, 3, 11, seed=22)
    out, _ = oracle.decode(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                           x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    ref = _brute_force_decode(x, 1e6, 1e-6)
    assert (out - ref).abs().max() < 1e-12


def test_decode_of_last_token_equals_last_prefill_row():
    """Prefill -> decode chunk equivalence (§20.9's chunked-cache check): the
    cache holds rounded normalised+rotated keys, so agreement is to bf16 rounding."""
    T, Hq, Hkv = 20, 4, 2
    x = inputs.prefill_inputs(1, T, Hq, Hkv, seed=23)
    full = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    khat = oracle.qknorm_rope(x["k"], x["k_gamma"], 1e6, 1e-6).to(torch.bfloat16)
    S = T + 3
    k_cache = torch.zeros((1, Hkv, S, D), dtype=torch.bfloat16)
    v_cache = torch.zeros((1, Hkv, S, D), dtype=torch.bfloat16)
    k_cache[0, :, : T - 1] = khat[0, : T - 1].transpose(0, 1)
    v_cache[0, :, : T - 1] = x["v"][0, : T - 1].transpose(0, 1)
    out, _ = oracle.decode(x["q"][:, T - 1], x["k"][:, T - 1], x["v"][:, T - 1], k_cache,
                           v_cache, [T - 1], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    assert (out[0] - full[0, T - 1]).abs().max() < 1e-2


def test_decode_rejects_context_overflow():
    x = inputs.decode_inputs(1, 2, 1, 4, 0, 1, seed=24, start_pos=[0])
    with pytest.raises(ValueError):
        oracle.decode(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], [4],
                      x["q_gamma"], x["k_gamma"], 1e6, 1e-6)


# ----------------------------------------------------------------------------
# Numbers the pages print
# ----------------------------------------------------------------------------

def test_kv_bytes_per_token_match_the_pages():
    with open(os.path.join(GOLDEN, "kv_cache_bytes_per_token.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        got = kv_cache_bytes_per_token(case["layers"], case["kv_heads"], case["head_dim"])
        assert got == case["bytes"]
        assert got == case["kib"] * 1024
    # "about 4.5 GiB" for 32K tokens of Qwen3-8B
    q3 = kv_cache_bytes_per_token(36, 8) * 32768 / 2 ** 30
    assert q3 == pytest.approx(gold["context_32k_tokens_gib"]["Qwen3-8B"], abs=0.05)


# ----------------------------------------------------------------------------
# Chunked prefill against a cache (§20.3: rectangular causal mask from
# pos_start; new keys rotated at their own positions, cached keys as stored)
# ----------------------------------------------------------------------------

def _brute_force_chunk(x, k_cache, v_cache, start_pos, theta, eps):
    q, k, v = (x[n].to(torch.float64).tolist() for n in ("q", "k", "v"))
    kc, vc = k_cache.to(torch.float64), v_cache.to(torch.float64)
    gq = x["q_gamma"].to(torch.float64).tolist()
    gk = x["k_gamma"].to(torch.float64).tolist()
    B, Tq, Hq, Hkv = len(q), len(q[0]), len(q[0][0]), len(k[0][0])
    g = Hq // Hkv

    def norm(row, gamma):
        inv = 1.0 / math.sqrt(math.fsum(e * e for e in row) / D + eps)
        return [row[c] * inv * gamma[c] for c in range(D)]

    def rotate(row, p):
        res = [0.0] * D
        for i in range(HALF):
            ang = p * theta ** (-2.0 * i / D)
            c, s = math.cos(ang), math.sin(ang)
            res[i] = c * row[i] - s * row[i + HALF]
            res[i + HALF] = s * row[i] + c * row[i + HALF]
        return res

    out = torch.zeros((B, Tq, Hq, D), dtype=torch.float64)
    for b in range(B):
        p0 = int(start_pos[b])
        for h in range(Hq):
            kv = ((h + 1) - 1) // g
            keys = [kc[b, kv, j].tolist() for j in range(p0)]
            vals = [vc[b, kv, j].tolist() for j in range(p0)]
            keys += [rotate(norm(k[b][t][kv], gk), p0 + t) for t in range(Tq)]
            vals += [v[b][t][kv] for t in range(Tq)]
            for t in range(Tq):
                qh = rotate(norm(q[b][t][h], gq), p0 + t)
                n = p0 + t + 1
                w = [math.exp(math.fsum(qh[c] * keys[j][c] for c in range(D)) / math.sqrt(D))
                     for j in range(n)]
                z = math.fsum(w)
                for c in range(D):
                    out[b, t, h, c] = math.fsum(w[j] * vals[j][c] for j in range(n)) / z
    return out


def test_chunk_matches_brute_force():
    B, Tq, Hq, Hkv, S = 2, 3, 4, 2, 12
    x = inputs.prefill_inputs(B, Tq, Hq, Hkv, seed=31)
    cache = inputs.decode_inputs(B, Hq, Hkv, S, 0, 1, seed=32, start_pos=[4, 7])
    out, _ = oracle.prefill_chunk(x["q"], x["k"], x["v"], cache["k_cache"], cache["v_cache"],
                                  [4, 7], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    ref = _brute_force_chunk(x, cache["k_cache"], cache["v_cache"], [4, 7], 1e6, 1e-6)
    assert (out - ref).abs().max() < 1e-12


def test_chunk_at_position_zero_is_prefill():
    B, T, Hq, Hkv, S = 2, 9, 8, 2, 16
    x = inputs.prefill_inputs(B, T, Hq, Hkv, seed=33)
    nan_cache = torch.full((B, Hkv, S, D), float("nan"), dtype=torch.bfloat16)
    out, k_rows = oracle.prefill_chunk(x["q"], x["k"], x["v"], nan_cache, nan_cache, [0, 0],
                                       x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    full = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    assert torch.equal(out, full)           # no cached row is read
    assert torch.equal(k_rows, oracle.qknorm_rope(x["k"], x["k_gamma"], 1e6, 1e-6))


def test_chunk_of_one_token_is_decode():
    B, Hq, Hkv, S = 3, 8, 4, 20
    y = inputs.decode_inputs(B, Hq, Hkv, S, 2, 19, seed=34)
    out, k_rows = oracle.prefill_chunk(y["q"][:, None], y["k_new"][:, None], y["v_new"][:, None],
                                       y["k_cache"], y["v_cache"], y["start_pos"], y["q_gamma"],
                                       y["k_gamma"], 1e6, 1e-6)
    dec, k_row = oracle.decode(y["q"], y["k_new"], y["v_new"], y["k_cache"], y["v_cache"],
                               y["start_pos"], y["q_gamma"], y["k_gamma"], 1e6, 1e-6)
    assert torch.equal(out[:, 0], dec)
    assert torch.equal(k_rows[:, 0], k_row)


def test_chunks_0_2_5_6_equal_one_prefill():
    """§20.9's chunked-cache check: chunks [0:2], [2:5], [5:6] through the cache
    give the full forward's outputs (to the bf16 rounding of cached keys)."""
    T, Hq, Hkv, S = 6, 4, 2, 8
    x = inputs.prefill_inputs(1, T, Hq, Hkv, seed=35)
    full = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    k_cache = torch.full((1, Hkv, S, D), float("nan"), dtype=torch.bfloat16)
    v_cache = torch.full((1, Hkv, S, D), float("nan"), dtype=torch.bfloat16)
    outs = []
    for lo, hi in [(0, 2), (2, 5), (5, 6)]:
        out, k_rows = oracle.prefill_chunk(x["q"][:, lo:hi], x["k"][:, lo:hi], x["v"][:, lo:hi],
                                           k_cache, v_cache, [lo], x["q_gamma"], x["k_gamma"],
                                           1e6, 1e-6)
        k_cache[0, :, lo:hi] = k_rows[0].transpose(0, 1).to(torch.bfloat16)
        v_cache[0, :, lo:hi] = x["v"][0, lo:hi].transpose(0, 1)
        outs.append(out)
    got = torch.cat(outs, dim=1)
    assert (got - full).abs().max() < 1e-2
    # the first chunk reads no cached row: exact
    assert torch.equal(outs[0], full[:, :2])


def test_chunk_rejects_overflow():
    x = inputs.prefill_inputs(1, 3, 2, 1, seed=36)
    cache = torch.zeros((1, 1, 4, D), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.prefill_chunk(x["q"], x["k"], x["v"], cache, cache, [2], x["q_gamma"],
                             x["k_gamma"], 1e6, 1e-6)
