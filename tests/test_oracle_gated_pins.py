"""Pins of the oracle's gated global-attention layer (Qwen3-Next / Qwen3.5) to
facts that do not come from the oracle itself.

Each test checks the oracle against a closed form, an invariant, a reduction
to the already pinned Qwen3 oracle, a value the pages print, or a separately
written brute force, so that a plausible slip (gamma used as the scale instead
of 1 + w, all d coordinates rotated, the frequency exponent over d instead of
d_r, the query/gate split done over the whole 2Hd vector instead of inside each
head, the gate applied before the softmax or without the sigmoid) fails at least
one of them.
"""
import json
import math
import os

import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import inputs
from qwen3_qk_norm_gb300.accounting import kv_cache_bytes_per_token

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_randn(*shape, seed=0, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def basis(d, i):
    e = torch.zeros(d, dtype=torch.float64)
    e[i] = 1.0
    return e


# ----------------------------------------------------------------------------
# g2: zero-centred RMSNorm, scale 1 + w ("Chapter 20" §20.4; Qwen3-Next section)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("eps", [1e-6, 1e-2])
def test_zc_norm_zero_weight_has_closed_form_rms(eps):
    """w = 0 (the initial weight) is a plain RMS normalisation: mean(y^2) =
    ms / (ms + eps) exactly."""
    x = bf16_randn(256, seed=1)
    y = oracle.zc_rmsnorm_row(x, torch.zeros(256, dtype=torch.bfloat16), eps)
    ms = math.fsum(v * v for v in x.to(torch.float64).tolist()) / 256
    assert float((y * y).mean()) == pytest.approx(ms / (ms + eps), rel=1e-13)


def test_zc_norm_minus_one_weight_is_zero_and_scale_is_one_plus_w():
    """w = -1 zeroes a coordinate; w = k/64 scales it by exactly 1 + k/64
    against w = 0 (a gamma-as-scale slip gives k/64 instead)."""
    x = bf16_randn(256, seed=2)
    w = torch.tensor([(k % 97 - 48) / 64 for k in range(256)], dtype=torch.float64)
    w[7] = -1.0
    y = oracle.zc_rmsnorm_row(x, w.to(torch.bfloat16), 1e-6)
    y0 = oracle.zc_rmsnorm_row(x, torch.zeros(256, dtype=torch.bfloat16), 1e-6)
    assert float(y[7]) == 0.0
    assert torch.allclose(y, y0 * (1.0 + w), rtol=1e-15, atol=0)


# ----------------------------------------------------------------------------
# g3: partial rotary ("Chapter 20" §20.4: only the first d_r coordinates turn,
# with d_r as the denominator of the frequency exponent)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("d,d_r", [(256, 64), (16, 4), (128, 0), (128, 128)])
def test_partial_rope_leaves_trailing_coordinates(d, d_r):
    y = torch.randn(d, dtype=torch.float64, generator=torch.Generator().manual_seed(3))
    for pos in [0, 1, 777, 262143]:
        r = oracle.partial_rope_row(y, d_r, pos, 1e7)
        assert torch.equal(r[d_r:], y[d_r:])
        h = d_r // 2
        if h:  # the rotated pairs keep their lengths
            assert torch.allclose(r[:h] ** 2 + r[h:d_r] ** 2, y[:h] ** 2 + y[h:d_r] ** 2,
                                  rtol=1e-13, atol=0)
    assert torch.equal(oracle.partial_rope_row(y, d_r, 0, 1e7), y)


@pytest.mark.parametrize("theta,pos,angle", [(math.pi ** -2, 1, math.pi),
                                             (1e4, 100, 1.0), (1e6, 1000, 1.0)])
def test_partial_rope_frequency_denominator_is_d_r(theta, pos, angle):
    """Pair i = d_r/4 turns by theta^(-1/2) per position when the exponent is
    2i/d_r: with theta = pi^-2 that is half a turn per position, with 1e4 it is
    1/100 rad, with 1e6 1/1000 rad. An exponent over d = 256 (1/8 instead of
    1/2) gives a different angle in each case."""
    d, d_r = 256, 64
    i, h = d_r // 4, d_r // 2
    lo = oracle.partial_rope_row(basis(d, i), d_r, pos, theta)
    hi = oracle.partial_rope_row(basis(d, i + h), d_r, pos, theta)
    exp_lo = torch.zeros(d, dtype=torch.float64)
    exp_lo[i], exp_lo[i + h] = math.cos(angle), math.sin(angle)
    exp_hi = torch.zeros(d, dtype=torch.float64)
    exp_hi[i], exp_hi[i + h] = -math.sin(angle), math.cos(angle)
    assert torch.allclose(lo, exp_lo, atol=1e-12, rtol=0)
    assert torch.allclose(hi, exp_hi, atol=1e-12, rtol=0)
    # pair 0 turns by exactly pos radians for every theta
    r0 = oracle.partial_rope_row(basis(d, 0), d_r, pos, theta)
    assert float(r0[0]) == pytest.approx(math.cos(pos), abs=1e-12)
    assert float(r0[h]) == pytest.approx(math.sin(pos), abs=1e-12)


@pytest.mark.parametrize("delta", [1, 5000, 200000])
def test_partial_rope_scores_depend_only_on_relative_position(delta):
    g = torch.Generator().manual_seed(4)
    q = torch.randn(256, dtype=torch.float64, generator=g)
    k = torch.randn(256, dtype=torch.float64, generator=g)
    for m, n in [(0, 5), (9, 2), (100, 3000)]:
        s0 = torch.dot(oracle.partial_rope_row(q, 64, m, 1e7), oracle.partial_rope_row(k, 64, n, 1e7))
        s1 = torch.dot(oracle.partial_rope_row(q, 64, m + delta, 1e7),
                       oracle.partial_rope_row(k, 64, n + delta, 1e7))
        assert float(s0) == pytest.approx(float(s1), abs=1e-9)


def test_partial_rope_rejects_odd_or_oversized_width():
    y = torch.zeros(16, dtype=torch.float64)
    for d_r in (3, 18, -2):
        with pytest.raises(ValueError):
            oracle.partial_rope_row(y, d_r, 1, 1e7)


# ----------------------------------------------------------------------------
# g1, g4, g5: per-head query/gate split, attention, sigmoid gate
# ----------------------------------------------------------------------------

def _qwen3_as_gated(x, gate_value):
    """The Qwen3 inputs x rewritten as a gated layer's inputs: the query of
    head h in qg[..., h, :d], a constant gate in qg[..., h, d:], w = gamma - 1
    (exact: the gammas below are 1 + k/64)."""
    B, T, Hq, d = x["q"].shape
    gate = torch.full((B, T, Hq, d), gate_value, dtype=torch.bfloat16)
    qg = torch.cat([x["q"], gate], dim=-1).contiguous()
    q_w = (x["q_gamma"].to(torch.float64) - 1.0).to(torch.bfloat16)
    k_w = (x["k_gamma"].to(torch.float64) - 1.0).to(torch.bfloat16)
    assert torch.equal(q_w.to(torch.float64) + 1.0, x["q_gamma"].to(torch.float64))
    assert torch.equal(k_w.to(torch.float64) + 1.0, x["k_gamma"].to(torch.float64))
    return qg, q_w, k_w


def _qwen3_inputs(B, T, Hq, Hkv, d, seed):
    x = inputs.prefill_inputs(B, T, Hq, Hkv, d=d, seed=seed)
    gm = torch.Generator().manual_seed(seed + 100)
    for name in ("q_gamma", "k_gamma"):
        k = torch.randint(-32, 32, (d,), generator=gm).to(torch.float64)
        x[name] = (1.0 + k / 64).to(torch.bfloat16)
    return x


@pytest.mark.parametrize("B,T,Hq,Hkv,d,theta", [(1, 7, 4, 2, 128, 1e6), (2, 5, 8, 2, 64, 1e7)])
def test_open_gate_full_rotary_reduces_to_qwen3(B, T, Hq, Hkv, d, theta):
    """sigmoid(100) is 1 in fp64, d_r = d rotates every coordinate and
    1 + (gamma - 1) = gamma: the gated layer is then the Qwen3 layer."""
    x = _qwen3_inputs(B, T, Hq, Hkv, d, seed=20)
    qg, q_w, k_w = _qwen3_as_gated(x, 100.0)
    got = oracle.gated_prefill(qg, x["k"], x["v"], q_w, k_w, d, theta, 1e-6)
    ref = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], theta, 1e-6)
    assert (got - ref).abs().max() < 1e-13


def test_zero_gate_halves_and_closed_gate_zeroes():
    """sigmoid(0) = 1/2 exactly; sigmoid(-100) < 4e-44."""
    x = _qwen3_inputs(1, 6, 4, 2, 64, seed=21)
    outs = {}
    for gv in (100.0, 0.0, -100.0):
        qg, q_w, k_w = _qwen3_as_gated(x, gv)
        outs[gv] = oracle.gated_prefill(qg, x["k"], x["v"], q_w, k_w, 16, 1e7, 1e-6)
    assert torch.equal(outs[0.0], outs[100.0] * 0.5)
    assert outs[-100.0].abs().max() < 4e-44 * outs[100.0].abs().max() + 1e-300


def test_gate_split_is_inside_each_head():
    """Closing the gate half of head 1 alone zeroes head 1's output and no
    other head's; opening it again restores it. A split of the whole 2*Hq*d
    vector into two halves would put head 1's gate elsewhere."""
    B, T, Hq, Hkv, d = 1, 5, 4, 2, 32
    x = _qwen3_inputs(B, T, Hq, Hkv, d, seed=22)
    qg, q_w, k_w = _qwen3_as_gated(x, 100.0)
    open_out = oracle.gated_prefill(qg, x["k"], x["v"], q_w, k_w, 8, 1e7, 1e-6)
    qg2 = qg.clone()
    qg2[:, :, 1, d:] = -100.0
    closed = oracle.gated_prefill(qg2, x["k"], x["v"], q_w, k_w, 8, 1e7, 1e-6)
    assert closed[:, :, 1].abs().max() < 1e-40
    for h in (0, 2, 3):
        assert torch.equal(closed[:, :, h], open_out[:, :, h])
    # the gate is elementwise over the head's d outputs: close one coordinate
    qg3 = qg.clone()
    qg3[:, :, 2, d + 5] = -100.0
    one = oracle.gated_prefill(qg3, x["k"], x["v"], q_w, k_w, 8, 1e7, 1e-6)
    assert one[:, :, 2, 5].abs().max() < 1e-40
    keep = torch.ones(d, dtype=torch.bool)
    keep[5] = False
    assert torch.equal(one[:, :, 2][..., keep], open_out[:, :, 2][..., keep])


def test_gate_acts_after_the_softmax():
    """The gate multiplies the attention output, so with every gate at 0 the
    row-0 output is exactly v_0 / 2 (row 0 attends to key 0 alone): a gate
    applied to the query or the scores would leave v_0 or change nothing."""
    x = inputs.gated_inputs(1, 4, 4, 2, d=32, seed=23)
    qg = x["qg"].clone()
    qg[..., 32:] = 0.0
    out = oracle.gated_prefill(qg, x["k"], x["v"], x["q_w"], x["k_w"], 8, 1e7, 1e-6)
    for h in range(4):
        assert torch.equal(out[0, 0, h], x["v"][0, 0, h // 2].to(torch.float64) * 0.5)


def _brute_force_gated(x, d_r, theta, eps):
    """Separately written brute force: the query/gate halves sliced with
    explicit per-head offsets into the flattened projection, the scale built
    as 1 + w, rotation by explicit 2x2 blocks over the first d_r coordinates,
    the logistic written as e^x / (1 + e^x), math-module sums. Tiny only."""
    qg = x["qg"].to(torch.float64)
    B, T, Hq, d2 = qg.shape
    d = d2 // 2
    flat = qg.reshape(B, T, Hq * d2).tolist()
    k, v = x["k"].to(torch.float64).tolist(), x["v"].to(torch.float64).tolist()
    sq = [1.0 + e for e in x["q_w"].to(torch.float64).tolist()]
    sk = [1.0 + e for e in x["k_w"].to(torch.float64).tolist()]
    Hkv = len(k[0][0])
    g = Hq // Hkv
    half = d_r // 2

    def norm(row, scale):
        inv = 1.0 / math.sqrt(math.fsum(e * e for e in row) / d + eps)
        return [row[c] * inv * scale[c] for c in range(d)]

    def rotate(row, p):
        res = list(row)
        for i in range(half):
            ang = p * theta ** (-2.0 * i / d_r)
            c, s = math.cos(ang), math.sin(ang)
            res[i] = c * row[i] - s * row[i + half]
            res[i + half] = s * row[i] + c * row[i + half]
        return res

    out = torch.zeros((B, T, Hq, d), dtype=torch.float64)
    for b in range(B):
        khat = [[rotate(norm(k[b][j][kv], sk), j) for kv in range(Hkv)] for j in range(T)]
        for i in range(T):
            for h in range(Hq):
                base = h * 2 * d
                query = flat[b][i][base:base + d]
                gate = flat[b][i][base + d:base + 2 * d]
                grp = h // g
                qh = rotate(norm(query, sq), i)
                w = [math.exp(math.fsum(qh[c] * khat[j][grp][c] for c in range(d)) / math.sqrt(d))
                     for j in range(i + 1)]
                z = math.fsum(w)
                for c in range(d):
                    o = math.fsum(w[j] * v[b][j][grp][c] for j in range(i + 1)) / z
                    e = math.exp(gate[c])
                    out[b, i, h, c] = o * e / (1.0 + e)
    return out


@pytest.mark.parametrize("B,T,Hq,Hkv,d,d_r,theta,seed", [
    (1, 6, 4, 2, 32, 8, 1e7, 30), (2, 4, 4, 1, 16, 4, 1e4, 31), (1, 5, 2, 2, 24, 24, 1e6, 32)])
def test_gated_prefill_matches_brute_force(B, T, Hq, Hkv, d, d_r, theta, seed):
    x = inputs.gated_inputs(B, T, Hq, Hkv, d=d, seed=seed)
    got = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], d_r, theta, 1e-6)
    ref = _brute_force_gated(x, d_r, theta, 1e-6)
    assert (got - ref).abs().max() < 1e-12


def test_gated_rows_equal_full_prefill_and_future_tokens_do_not_matter():
    B, T, Hq, Hkv, d = 2, 21, 4, 2, 256
    x = inputs.gated_inputs(B, T, Hq, Hkv, d=d, seed=33)
    full = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    rows = torch.tensor([[0, 0, 0], [1, 20, 3], [0, 13, 2], [1, 7, 1]], dtype=torch.int32)
    got = oracle.gated_prefill_rows(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6,
                                    rows)
    for n, (b, t, h) in enumerate(rows.tolist()):
        assert torch.equal(got[n], full[b, t, h])
    # causality: changing token 15 onwards leaves rows 0..14 unchanged
    y = {k: t.clone() for k, t in x.items()}
    for name in ("qg", "k", "v"):
        y[name][:, 15:] = bf16_randn(*y[name][:, 15:].shape, seed=34)
    other = oracle.gated_prefill(y["qg"], y["k"], y["v"], y["q_w"], y["k_w"], 64, 1e7, 1e-6)
    assert torch.equal(other[:, :15], full[:, :15])
    assert not torch.equal(other[:, 15:], full[:, 15:])


def test_gated_rejects_bad_shapes():
    x = inputs.gated_inputs(1, 3, 4, 2, d=16, seed=35)
    with pytest.raises(ValueError):
        oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 5, 1e7, 1e-6)
    with pytest.raises(ValueError):
        oracle.gated_prefill(x["qg"][..., :24].contiguous(), x["k"], x["v"], x["q_w"],
                             x["k_w"], 4, 1e7, 1e-6)


# ----------------------------------------------------------------------------
# Numbers the pages print
# ----------------------------------------------------------------------------

def test_qwen3_next_global_kv_bytes_match_the_pages():
    with open(os.path.join(GOLDEN, "qwen3_next_global_kv_bytes.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        got = kv_cache_bytes_per_token(case["layers"], case["kv_heads"], case["head_dim"])
        assert got == case["bytes"] == case["kib"] * 1024
    ctx = gold["context_100k_tokens_gib"]
    assert kv_cache_bytes_per_token(36, 8) * 100000 / 2 ** 30 == pytest.approx(
        ctx["Qwen3-8B"], abs=0.05)
    assert kv_cache_bytes_per_token(12, 2, 256) * 100000 / 2 ** 30 == pytest.approx(
        ctx["Qwen3-Next-80B-A3B global layers"], abs=0.05)


def test_gated_qknorm_rope_rows_are_the_pinned_steps():
    """The row-array form applies g2 then g3 to the first d elements of each
    row (the query half of a query/gate block), at position pos0 + t."""
    x = inputs.gated_inputs(2, 3, 2, 1, d=32, seed=36)
    got = oracle.gated_qknorm_rope(x["qg"], x["q_w"], 32, 8, 1e7, 1e-6, pos0=4)
    for b in range(2):
        for t in range(3):
            for h in range(2):
                ref = oracle.partial_rope_row(
                    oracle.zc_rmsnorm_row(x["qg"][b, t, h, :32], x["q_w"], 1e-6), 8, 4 + t, 1e7)
                assert torch.equal(got[b, t, h], ref)


# ----------------------------------------------------------------------------
# Gated decode (§20.3's cache protocol on the gated layer)
# ----------------------------------------------------------------------------

def test_gated_decode_at_position_zero_is_gated_v_new():
    """One key: the attention output is v_new, so z = v_new * sigmoid(gate)."""
    B, Hq, Hkv, S, d = 2, 4, 2, 3, 32
    x = inputs.gated_decode_inputs(B, Hq, Hkv, S, 0, 1, d=d, seed=40, start_pos=[0, 0])
    out, k_row = oracle.gated_decode(x["qg"], x["k_new"], x["v_new"], x["k_cache"],
                                     x["v_cache"], x["start_pos"], x["q_w"], x["k_w"], 8, 1e7,
                                     1e-6)
    for b in range(B):
        for h in range(Hq):
            gate = x["qg"][b, h, d:].to(torch.float64)
            ref = x["v_new"][b, h // 2].to(torch.float64) / (1.0 + torch.exp(-gate))
            assert torch.allclose(out[b, h], ref, atol=1e-15, rtol=1e-15)
        for kv in range(Hkv):  # RoPE at position 0 is the identity
            assert torch.equal(k_row[b, kv], oracle.zc_rmsnorm_row(x["k_new"][b, kv], x["k_w"],
                                                                   1e-6))


def _brute_force_gated_decode(x, d_r, theta, eps):
    qg = x["qg"].to(torch.float64)
    B, Hq, d2 = qg.shape
    d = d2 // 2
    kn, vn = x["k_new"].to(torch.float64).tolist(), x["v_new"].to(torch.float64).tolist()
    kc, vc = x["k_cache"].to(torch.float64), x["v_cache"].to(torch.float64)
    sq = [1.0 + e for e in x["q_w"].to(torch.float64).tolist()]
    sk = [1.0 + e for e in x["k_w"].to(torch.float64).tolist()]
    Hkv = len(kn[0])
    g, half = Hq // Hkv, d_r // 2

    def norm(row, scale):
        inv = 1.0 / math.sqrt(math.fsum(e * e for e in row) / d + eps)
        return [row[c] * inv * scale[c] for c in range(d)]

    def rotate(row, p):
        res = list(row)
        for i in range(half):
            ang = p * theta ** (-2.0 * i / d_r)
            c, s = math.cos(ang), math.sin(ang)
            res[i] = c * row[i] - s * row[i + half]
            res[i + half] = s * row[i] + c * row[i + half]
        return res

    out = torch.zeros((B, Hq, d), dtype=torch.float64)
    flat = qg.reshape(B, Hq * d2).tolist()
    for b in range(B):
        p = int(x["start_pos"][b])
        for h in range(Hq):
            kv = h // g
            keys = [kc[b, kv, j].tolist() for j in range(p)] + [rotate(norm(kn[b][kv], sk), p)]
            vals = [vc[b, kv, j].tolist() for j in range(p)] + [vn[b][kv]]
            query = flat[b][h * d2:h * d2 + d]
            gate = flat[b][h * d2 + d:h * d2 + 2 * d]
            qh = rotate(norm(query, sq), p)
            w = [math.exp(math.fsum(qh[c] * kr[c] for c in range(d)) / math.sqrt(d))
                 for kr in keys]
            z = math.fsum(w)
            for c in range(d):
                o = math.fsum(w[j] * vals[j][c] for j in range(len(keys))) / z
                out[b, h, c] = o * math.exp(gate[c]) / (1.0 + math.exp(gate[c]))
    return out


def test_gated_decode_matches_brute_force_with_cache_used_as_stored():
    x = inputs.gated_decode_inputs(2, 4, 2, 12, 3, 11, d=32, seed=41)
    out, _ = oracle.gated_decode(x["qg"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                                 x["start_pos"], x["q_w"], x["k_w"], 8, 1e7, 1e-6)
    ref = _brute_force_gated_decode(x, 8, 1e7, 1e-6)
    assert (out - ref).abs().max() < 1e-12


def test_gated_decode_of_last_token_equals_last_prefill_row():
    """Prefill -> decode equivalence on the gated layer: the cache holds the
    rounded normalised+rotated keys, so agreement is to bf16 rounding."""
    T, Hq, Hkv, d = 20, 4, 2, 256
    x = inputs.gated_inputs(1, T, Hq, Hkv, d=d, seed=42)
    full = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    khat = oracle.gated_qknorm_rope(x["k"], x["k_w"], d, 64, 1e7, 1e-6).to(torch.bfloat16)
    S = T + 3
    k_cache = torch.zeros((1, Hkv, S, d), dtype=torch.bfloat16)
    v_cache = torch.zeros((1, Hkv, S, d), dtype=torch.bfloat16)
    k_cache[0, :, : T - 1] = khat[0, : T - 1].transpose(0, 1)
    v_cache[0, :, : T - 1] = x["v"][0, : T - 1].transpose(0, 1)
    out, k_row = oracle.gated_decode(x["qg"][:, T - 1].contiguous(), x["k"][:, T - 1].contiguous(),
                                     x["v"][:, T - 1].contiguous(), k_cache, v_cache, [T - 1],
                                     x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    assert (out[0] - full[0, T - 1]).abs().max() < 1e-2
    ref_k = oracle.gated_qknorm_rope(x["k"], x["k_w"], d, 64, 1e7, 1e-6)[0, T - 1]
    assert torch.equal(k_row[0], ref_k)


def test_gated_decode_rejects_context_overflow():
    x = inputs.gated_decode_inputs(1, 2, 1, 4, 0, 1, d=16, seed=43, start_pos=[0])
    with pytest.raises(ValueError):
        oracle.gated_decode(x["qg"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], [4],
                            x["q_w"], x["k_w"], 4, 1e7, 1e-6)


# ----------------------------------------------------------------------------
# Gated chunk against a cache (§20.3: rectangular causal mask from pos_start)
# ----------------------------------------------------------------------------

def test_gated_chunk_at_position_zero_is_gated_prefill():
    x = inputs.gated_inputs(2, 9, 4, 2, d=32, seed=50)
    kc = torch.zeros((2, 2, 12, 32), dtype=torch.bfloat16)
    out, k_rows = oracle.gated_prefill_chunk(x["qg"], x["k"], x["v"], kc, kc.clone(), [0, 0],
                                             x["q_w"], x["k_w"], 8, 1e7, 1e-6)
    ref = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 8, 1e7, 1e-6)
    assert torch.equal(out, ref)
    assert torch.equal(k_rows, oracle.gated_qknorm_rope(x["k"], x["k_w"], 32, 8, 1e7, 1e-6))


def test_gated_chunk_of_one_token_is_gated_decode():
    x = inputs.gated_decode_inputs(2, 4, 2, 16, 3, 12, d=32, seed=51)
    out, _ = oracle.gated_prefill_chunk(x["qg"][:, None], x["k_new"][:, None],
                                        x["v_new"][:, None], x["k_cache"], x["v_cache"],
                                        x["start_pos"], x["q_w"], x["k_w"], 8, 1e7, 1e-6)
    ref, _ = oracle.gated_decode(x["qg"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                                 x["start_pos"], x["q_w"], x["k_w"], 8, 1e7, 1e-6)
    assert torch.equal(out[:, 0], ref)


def test_gated_chunks_in_sequence_equal_one_prefill():
    """Chunks [0:2], [2:5], [5:6] of a prompt through a bf16 cache give the
    full prefill's rows (the first chunk exactly, the later ones to the
    rounding of the cached keys)."""
    T, Hq, Hkv, d = 6, 4, 2, 32
    x = inputs.gated_inputs(1, T, Hq, Hkv, d=d, seed=52)
    full = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 8, 1e7, 1e-6)
    kc = torch.zeros((1, Hkv, 8, d), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    for i, (a, b) in enumerate([(0, 2), (2, 5), (5, 6)]):
        part, k_rows = oracle.gated_prefill_chunk(
            x["qg"][:, a:b].contiguous(), x["k"][:, a:b].contiguous(), x["v"][:, a:b].contiguous(),
            kc, vc, [a], x["q_w"], x["k_w"], 8, 1e7, 1e-6)
        if i == 0:
            assert torch.equal(part, full[:, a:b])
        else:
            assert (part - full[:, a:b]).abs().max() < 1e-2
        kc[0, :, a:b] = k_rows[0].transpose(0, 1).to(torch.bfloat16)
        vc[0, :, a:b] = x["v"][0, a:b].transpose(0, 1)


def test_gated_chunk_rejects_overflow():
    x = inputs.gated_inputs(1, 3, 2, 1, d=16, seed=53)
    kc = torch.zeros((1, 1, 4, 16), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.gated_prefill_chunk(x["qg"], x["k"], x["v"], kc, kc, [2], x["q_w"], x["k_w"], 4,
                                   1e7, 1e-6)
