"""Gated global attention of Qwen3-Next / Qwen3.5 (K5 prologue + K6 attention)
on the GPU against the fp64 oracle, via the C ABI."""
import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import binding, inputs
from qwen3_qk_norm_gb300.inputs import WORKLOADS
from gpu_util import assert_close_attention, assert_within_one_ulp

pytestmark = pytest.mark.gpu

D = 256


def run_gated(x, d_r, theta, eps=1e-6, workspace=None):
    d = {k: t.cuda() for k, t in x.items()}
    out = binding.gated_prefill(d["qg"], d["k"], d["v"], d["q_w"], d["k_w"], d_r, theta, eps,
                                workspace=workspace)
    torch.cuda.synchronize()
    return out


def workspace_views(ws, B, T, Hq, Hkv):
    """Qhat [B,T,Hq,256] and Khat [B,Hkv,T,256] inside a gated workspace."""
    q_bytes = B * T * Hq * D * 2
    k_off = 256 + ((q_bytes + 255) // 256) * 256
    qhat = ws[256:256 + q_bytes].view(torch.bfloat16).view(B, T, Hq, D)
    khat = ws[k_off:k_off + B * T * Hkv * D * 2].view(torch.bfloat16).view(B, Hkv, T, D)
    return qhat, khat


@pytest.mark.parametrize("B,T,Hq,Hkv,d_r,theta", [(1, 37, 8, 2, 64, 1e7), (2, 20, 16, 2, 64, 1e7),
                                                  (1, 9, 4, 4, 256, 1e6), (1, 5, 4, 2, 0, 1e7),
                                                  (1, 70000, 1, 1, 64, 1e7)])
def test_gated_prologue_within_one_ulp(cuda_lib, B, T, Hq, Hkv, d_r, theta):
    """Zero-centred norm + partial RoPE: one rounding of the fp32 result, so at
    most one bf16 ulp from the exact value (positions up to 70000)."""
    x = inputs.gated_inputs(B, T, Hq, Hkv, seed=T + Hq)
    d = {k: t.cuda() for k, t in x.items()}
    ws = torch.zeros(binding.gated_prefill_workspace_size(B, T, Hq, Hkv), dtype=torch.uint8,
                     device="cuda")
    binding.gated_prefill_prologue(d["qg"], d["k"], d["q_w"], d["k_w"], d_r, theta, 1e-6, ws)
    torch.cuda.synchronize()
    qhat, khat = workspace_views(ws, B, T, Hq, Hkv)
    ref_q = oracle.gated_qknorm_rope(x["qg"], x["q_w"], D, d_r, theta, 1e-6)
    ref_k = oracle.gated_qknorm_rope(x["k"], x["k_w"], D, d_r, theta, 1e-6)
    assert_within_one_ulp(qhat, ref_q, "qhat")
    assert_within_one_ulp(khat.permute(0, 2, 1, 3), ref_k, "khat")
    # the bound the attention kernel's fixed-shift softmax relies on
    bound = float(ws[8:12].view(torch.float32).item())
    gq = float((1.0 + x["q_w"].double()).abs().max())
    gk = float((1.0 + x["k_w"].double()).abs().max())
    assert bound == pytest.approx(16 * gq * gk * 1.4426950408889634, rel=1e-6)


# small shapes: several M tiles and KV tiles, ragged tails, every g
@pytest.mark.parametrize("B,T,Hq,Hkv,d_r,theta", [
    (1, 1, 8, 2, 64, 1e7),      # a single token
    (1, 2, 2, 2, 64, 1e7),      # g = 1
    (1, 63, 8, 2, 64, 1e7),     # one KV tile minus one
    (2, 65, 4, 2, 64, 1e7),     # one KV tile plus one, B > 1
    (1, 200, 16, 1, 64, 1e7),   # g = 16
    (1, 300, 16, 2, 64, 1e7),   # g = 8, Qwen3-Next heads
    (2, 150, 8, 8, 64, 1e6),    # g = 1, ragged
    (1, 129, 8, 4, 256, 1e6),   # full rotary
    (1, 100, 4, 2, 0, 1e7),     # no rotary
    (1, 180, 24, 4, 64, 1e7),   # g = 6 (Qwen3.5-27B heads): 126-row tiles, 2 padding rows
    (2, 90, 24, 2, 64, 1e7),    # g = 12 (Qwen3.8-Flash-Next heads): 120-row tiles
])
def test_gated_prefill_small_shapes(cuda_lib, B, T, Hq, Hkv, d_r, theta):
    x = inputs.gated_inputs(B, T, Hq, Hkv, seed=B * 1000 + T)
    ref = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], d_r, theta, 1e-6)
    assert_close_attention(run_gated(x, d_r, theta), ref,
                           f"gated B{B} T{T} Hq{Hq} Hkv{Hkv} d_r{d_r}")


def test_gated_qwen35_08b_t300_full(cuda_lib):
    w = WORKLOADS["qwen3.5-0.8b-gated-b1-t300"]
    x = inputs.workload_inputs(w)
    ref = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], w.d_r, w.theta, w.eps)
    assert_close_attention(run_gated(x, w.d_r, w.theta), ref, w.name)


@pytest.mark.parametrize("wmax", [0.5, 1.2, 2.5])  # bound <= 52, ~112, ~283 (log2 units)
def test_gated_both_softmax_paths(cuda_lib, wmax):
    """The norm bounds the logits by 16 max|1 + w_q| max|1 + w_k|; above the
    kernel's limit the online-max path runs. Both must match the oracle."""
    x = inputs.gated_inputs(1, 300, 8, 2, seed=int(wmax * 10))
    g = torch.Generator().manual_seed(78)
    x["q_w"] = (torch.rand(D, generator=g) * 2 * wmax - wmax).to(torch.bfloat16)
    x["k_w"] = (torch.rand(D, generator=g) * 2 * wmax - wmax).to(torch.bfloat16)
    ref = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    assert_close_attention(run_gated(x, 64, 1e7), ref, f"w max {wmax}")


def test_gated_closed_and_open_gates(cuda_lib):
    """Gates at -100 give exact zeros; the output is elementwise in the gate."""
    x = inputs.gated_inputs(1, 90, 8, 2, seed=9)
    x["qg"][:, :, 3, D:] = -100.0
    ref = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    out = run_gated(x, 64, 1e7)
    assert bool((out[:, :, 3] == 0).all())
    assert_close_attention(out, ref, "closed gate of head 3")


def test_gated_halves_equal_whole_call(cuda_lib):
    B, T, Hq, Hkv = 2, 150, 16, 2
    x = inputs.gated_inputs(B, T, Hq, Hkv, seed=10)
    d = {k: t.cuda() for k, t in x.items()}
    whole = run_gated(x, 64, 1e7)
    ws = torch.empty(binding.gated_prefill_workspace_size(B, T, Hq, Hkv), dtype=torch.uint8,
                     device="cuda")
    binding.gated_prefill_prologue(d["qg"], d["k"], d["q_w"], d["k_w"], 64, 1e7, 1e-6, ws)
    out = torch.empty((B, T, Hq, D), dtype=torch.bfloat16, device="cuda")
    binding.gated_prefill_attention(d["qg"], d["v"], out, ws)
    torch.cuda.synchronize()
    assert binding.last_device_error(ws) == binding.Q3A_OK
    assert torch.equal(out, whole)


def test_gated_is_deterministic(cuda_lib):
    x = inputs.gated_inputs(1, 260, 16, 2, seed=11)
    a = run_gated(x, 64, 1e7)
    b = run_gated(x, 64, 1e7)
    assert torch.equal(a, b)


def test_gated_prefill_fill_writes_caches_and_matches_prefill(cuda_lib):
    """The cache-filling prefill gives the plain gated prefill's output bits and
    leaves the normalised, rotated keys and the values in cache rows 0..T-1."""
    B, T, Hq, Hkv, S = 2, 170, 16, 2, 300
    x = inputs.gated_inputs(B, T, Hq, Hkv, seed=15)
    d = {k: t.cuda() for k, t in x.items()}
    plain = binding.gated_prefill(d["qg"], d["k"], d["v"], d["q_w"], d["k_w"], 64, 1e7, 1e-6)
    kc = torch.full((B, Hkv, S, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    out = binding.gated_prefill_fill(d["qg"], d["k"], d["v"], kc, vc, d["q_w"], d["k_w"], 64,
                                     1e7, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(out, plain)
    ref_k = oracle.gated_qknorm_rope(x["k"], x["k_w"], D, 64, 1e7, 1e-6)
    assert_within_one_ulp(kc[:, :, :T].permute(0, 2, 1, 3), ref_k, "cached keys")
    assert torch.equal(vc[:, :, :T].cpu(), x["v"].transpose(1, 2))
    assert bool(torch.isnan(kc[:, :, T:].float()).all()) and bool(torch.isnan(vc[:, :, T:].float()).all())


def test_gated_prefill_fill_then_decode_continues_the_sequence(cuda_lib):
    """Prompt through q3a_gated_prefill_fill, then three q3a_gated_decode steps
    on the caches it filled: each step's output is the oracle's prefill row of
    the grown sequence (to the bf16 rounding of the cached keys)."""
    T0, steps, Hq, Hkv = 257, 3, 8, 2
    x = inputs.gated_inputs(1, T0 + steps, Hq, Hkv, seed=16)
    full = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    d = {k: t.cuda() for k, t in x.items()}
    S = 512
    kc = torch.full((1, Hkv, S, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    out = binding.gated_prefill_fill(d["qg"][:, :T0].contiguous(), d["k"][:, :T0].contiguous(),
                                     d["v"][:, :T0].contiguous(), kc, vc, d["q_w"], d["k_w"], 64,
                                     1e7, 1e-6)
    torch.cuda.synchronize()
    assert_close_attention(out, full[:, :T0], "prompt")
    for s in range(steps):
        t = T0 + s
        o = binding.gated_decode(d["qg"][:, t].contiguous(), d["k"][:, t].contiguous(),
                                 d["v"][:, t].contiguous(), kc, vc, [t], d["q_w"], d["k_w"], 64,
                                 1e7, 1e-6)
        torch.cuda.synchronize()
        assert_close_attention(o[0], full[0, t], f"decode step {s}")


# ----------------------------------------------------------------------------
# Gated chunk against the caches (q3a_gated_prefill_chunk)
# ----------------------------------------------------------------------------

def gated_chunk_case(B, Tq, Hq, Hkv, S, start_pos, seed):
    """Chunk inputs plus caches whose rows 0..start_pos[b]-1 hold random keys
    and values and whose later rows are NaN."""
    x = inputs.gated_inputs(B, Tq, Hq, Hkv, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    kc = torch.randn((B, Hkv, S, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, S, D), generator=g).to(torch.bfloat16)
    for b, p in enumerate(start_pos):
        kc[b, :, p:] = float("nan")
        vc[b, :, p:] = float("nan")
    return x, kc, vc


@pytest.mark.parametrize("Tq,Hq,Hkv,d_r,start_pos", [
    (37, 16, 2, 64, [0, 1, 127, 128, 1000]),   # Qwen3-Next heads; tile boundaries
    (300, 8, 2, 64, [5, 700]),                 # several pair tiles, ragged tail
    (1, 16, 2, 64, [0, 300, 2047]),            # one token per sequence
    (130, 32, 2, 64, [64, 200]),               # g = 16
    (50, 4, 4, 256, [90]),                     # g = 1, full rotary
    (70, 24, 4, 64, [33, 513]),                # g = 6
    (40, 24, 2, 0, [129, 7]),                  # g = 12, no rotary
])
def test_gated_chunk_matches_oracle_and_appends(cuda_lib, Tq, Hq, Hkv, d_r, start_pos):
    B, S = len(start_pos), 2400
    x, kc, vc = gated_chunk_case(B, Tq, Hq, Hkv, S, start_pos, seed=Tq + Hq + d_r)
    d = {k: t.cuda() for k, t in x.items()}
    kc_d, vc_d = kc.cuda(), vc.cuda()
    out = binding.gated_prefill_chunk(d["qg"], d["k"], d["v"], kc_d, vc_d, start_pos, d["q_w"],
                                      d["k_w"], d_r, 1e7, 1e-6)
    torch.cuda.synchronize()
    ref, k_rows = oracle.gated_prefill_chunk(x["qg"], x["k"], x["v"], kc, vc, start_pos,
                                             x["q_w"], x["k_w"], d_r, 1e7, 1e-6)
    assert bool(torch.isfinite(out).all())
    assert_close_attention(out, ref, f"gated chunk Tq{Tq} Hq{Hq} Hkv{Hkv}")
    kc_o, vc_o = kc_d.cpu(), vc_d.cpu()
    for b, p in enumerate(start_pos):
        assert_within_one_ulp(kc_o[b, :, p:p + Tq].transpose(0, 1), k_rows[b], f"keys b{b}")
        assert torch.equal(vc_o[b, :, p:p + Tq].view(torch.int16),
                           x["v"][b].transpose(0, 1).view(torch.int16))
        assert torch.equal(kc_o[b, :, :p].view(torch.int16), kc[b, :, :p].view(torch.int16))
        assert bool(torch.isnan(kc_o[b, :, p + Tq:].float()).all())
        assert bool(torch.isnan(vc_o[b, :, p + Tq:].float()).all())


def test_gated_chunk_at_zero_is_the_filling_prefill(cuda_lib):
    """Every start position 0: the chunk gives q3a_gated_prefill_fill's output
    and caches bit for bit (the same logit-bound path, the same tiles)."""
    B, T, Hq, Hkv, S = 2, 170, 16, 2, 300
    x = inputs.gated_inputs(B, T, Hq, Hkv, seed=21)
    d = {k: t.cuda() for k, t in x.items()}
    kc1 = torch.full((B, Hkv, S, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc1, kc2, vc2 = kc1.clone(), kc1.clone(), kc1.clone()
    fill = binding.gated_prefill_fill(d["qg"], d["k"], d["v"], kc1, vc1, d["q_w"], d["k_w"], 64,
                                      1e7, 1e-6)
    chunk = binding.gated_prefill_chunk(d["qg"], d["k"], d["v"], kc2, vc2, [0, 0], d["q_w"],
                                        d["k_w"], 64, 1e7, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(chunk, fill)
    assert torch.equal(kc1.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc1.view(torch.int16), vc2.view(torch.int16))


def test_gated_chunks_in_sequence_equal_one_prefill(cuda_lib):
    """A 600-token prompt as chunks [0:130], [130:300], [300:301], [301:600]
    through the caches: every chunk's rows match the oracle's one-shot gated
    prefill of the whole prompt (to the cache's bf16 rounding of the keys)."""
    T, Hq, Hkv = 600, 16, 2
    x = inputs.gated_inputs(1, T, Hq, Hkv, seed=22)
    full = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    d = {k: t.cuda() for k, t in x.items()}
    kc = torch.full((1, Hkv, 1024, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    for a, e in [(0, 130), (130, 300), (300, 301), (301, 600)]:
        out = binding.gated_prefill_chunk(d["qg"][:, a:e].contiguous(), d["k"][:, a:e].contiguous(),
                                          d["v"][:, a:e].contiguous(), kc, vc, [a], d["q_w"],
                                          d["k_w"], 64, 1e7, 1e-6)
        torch.cuda.synchronize()
        assert_close_attention(out, full[:, a:e], f"chunk [{a}:{e}]")


def test_gated_chunk_erange_writes_nothing(cuda_lib):
    x, kc, vc = gated_chunk_case(2, 10, 16, 2, 64, [3, 60], seed=23)
    d = {k: t.cuda() for k, t in x.items()}
    kc_d, vc_d = kc.cuda(), vc.cuda()
    out = torch.full((2, 10, 16, D), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.Q3AError) as err:
        binding.gated_prefill_chunk(d["qg"], d["k"], d["v"], kc_d, vc_d, [3, 60], d["q_w"],
                                    d["k_w"], 64, 1e7, 1e-6, out=out)
    assert err.value.status == binding.Q3A_ERANGE
    torch.cuda.synchronize()
    assert torch.equal(kc_d.cpu().view(torch.int16), kc.view(torch.int16))
    assert bool((out == 3.0).all())


def test_gated_more_items_than_pairs_full_parity(cuda_lib):
    """80 pair items (32-token pair tiles of 4 KV groups) on a GPU with fewer
    than 80 pairs of SMs: some persistent pairs take a second item. Every
    output row against the oracle."""
    x = inputs.gated_inputs(2, 640, 16, 2, seed=32)
    ref = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    assert_close_attention(run_gated(x, 64, 1e7), ref, "80 pair items")


def test_gated_chunk_more_items_than_pairs_with_tails(cuda_lib):
    """100 pair items (ten 32-token pair tiles for each of 10 (b, kv) groups)
    on persistent pairs, so several pairs take more than one item, each
    sequence's valid keys ending inside a 128-key tile of NaN-poisoned cache
    rows. Every output row and appended row against the oracle."""
    B, Tq, Hq, Hkv, S = 5, 320, 16, 2, 2000
    start_pos = [33, 400, 777, 1200, 1500]
    x, kc, vc = gated_chunk_case(B, Tq, Hq, Hkv, S, start_pos, seed=34)
    d = {k: t.cuda() for k, t in x.items()}
    kc_d, vc_d = kc.cuda(), vc.cuda()
    out = binding.gated_prefill_chunk(d["qg"], d["k"], d["v"], kc_d, vc_d, start_pos, d["q_w"],
                                      d["k_w"], 64, 1e7, 1e-6)
    torch.cuda.synchronize()
    ref, k_rows = oracle.gated_prefill_chunk(x["qg"], x["k"], x["v"], kc, vc, start_pos,
                                             x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    assert bool(torch.isfinite(out).all())
    assert_close_attention(out, ref, "100 gated chunk items with tails")
    kc_o = kc_d.cpu()
    for b, p in enumerate(start_pos):
        assert_within_one_ulp(kc_o[b, :, p:p + Tq].transpose(0, 1), k_rows[b], f"keys b{b}")


@pytest.mark.parametrize("scale,expect_error", [(1.5, False), (1.0e4, True)])
def test_gated_chunk_cache_above_the_bound(cuda_lib, scale, expect_error):
    """As for the Qwen3 chunk: cached keys 1.5 times longer than this library
    writes them still give the oracle's output (the shift cancels); keys 10^4
    times too long overflow the softmax sum and the call reports Q3A_EINVAL."""
    B, Tq, Hq, Hkv, S = 2, 40, 16, 2, 600
    start_pos = [300, 450]
    x, kc, vc = gated_chunk_case(B, Tq, Hq, Hkv, S, start_pos, seed=36)
    for b, p in enumerate(start_pos):
        kc[b, :, :p] = (kc[b, :, :p].float() * scale).to(torch.bfloat16)
    d = {k: t.cuda() for k, t in x.items()}
    kc_d, vc_d = kc.cuda(), vc.cuda()
    ws = torch.empty(binding.gated_prefill_chunk_workspace_size(B, Tq, Hq, Hkv),
                     dtype=torch.uint8, device="cuda")
    out = binding.gated_prefill_chunk(d["qg"], d["k"], d["v"], kc_d, vc_d, start_pos, d["q_w"],
                                      d["k_w"], 64, 1e7, 1e-6, workspace=ws)
    torch.cuda.synchronize()
    status = binding.last_device_error(ws)
    if expect_error:
        assert status == binding.Q3A_EINVAL
    else:
        assert status == binding.Q3A_OK
        ref, _ = oracle.gated_prefill_chunk(x["qg"], x["k"], x["v"], kc, vc, start_pos,
                                            x["q_w"], x["k_w"], 64, 1e7, 1e-6)
        assert_close_attention(out, ref, "gated cache keys x1.5")


@pytest.mark.parametrize("d_r", [16, 48, 128, 240])
def test_gated_rotary_widths(cuda_lib, d_r):
    """Every rotary width the entry points accept is a multiple of 16: the
    prologue's lane layout (d_r / 8 lanes holding rotated pairs) and the decode
    kernel's rotation take other shapes than at 64 and 256. Prologue rows to
    one bf16 ulp, prefill and decode outputs against the oracle."""
    B, T, Hq, Hkv = 2, 45, 8, 2
    x = inputs.gated_inputs(B, T, Hq, Hkv, seed=40 + d_r)
    d = {k: t.cuda() for k, t in x.items()}
    ws = torch.zeros(binding.gated_prefill_workspace_size(B, T, Hq, Hkv), dtype=torch.uint8,
                     device="cuda")
    binding.gated_prefill_prologue(d["qg"], d["k"], d["q_w"], d["k_w"], d_r, 1e7, 1e-6, ws)
    torch.cuda.synchronize()
    qhat, khat = workspace_views(ws, B, T, Hq, Hkv)
    assert_within_one_ulp(qhat, oracle.gated_qknorm_rope(x["qg"], x["q_w"], D, d_r, 1e7, 1e-6),
                          f"qhat d_r {d_r}")
    assert_within_one_ulp(khat.permute(0, 2, 1, 3),
                          oracle.gated_qknorm_rope(x["k"], x["k_w"], D, d_r, 1e7, 1e-6),
                          f"khat d_r {d_r}")
    out = run_gated(x, d_r, 1e7)
    ref = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], d_r, 1e7, 1e-6)
    assert_close_attention(out, ref, f"gated prefill d_r {d_r}")
    y = inputs.gated_decode_inputs(3, Hq, Hkv, 600, 0, 1, seed=41 + d_r, start_pos=[0, 129, 599])
    dy = {k: (t.cuda() if k != "start_pos" else t) for k, t in y.items()}
    o2 = binding.gated_decode(dy["qg"], dy["k_new"], dy["v_new"], dy["k_cache"], dy["v_cache"],
                              y["start_pos"], dy["q_w"], dy["k_w"], d_r, 1e7, 1e-6)
    torch.cuda.synchronize()
    r2, _ = oracle.gated_decode(y["qg"], y["k_new"], y["v_new"], y["k_cache"], y["v_cache"],
                                y["start_pos"], y["q_w"], y["k_w"], d_r, 1e7, 1e-6)
    assert_close_attention(o2, r2, f"gated decode d_r {d_r}")


def test_gated_output_only_16_byte_aligned(cuda_lib):
    """32-byte stores when the output allows them, 16-byte ones otherwise: an
    output that starts 16 bytes into a buffer gets the same bits."""
    B, T, Hq, Hkv = 1, 150, 16, 2
    x = {k: t.cuda() for k, t in inputs.gated_inputs(B, T, Hq, Hkv, seed=19).items()}
    full = binding.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    buf = torch.empty(B * T * Hq * D + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(B, T, Hq, D)
    assert out.data_ptr() % 32 == 16
    binding.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, full)
