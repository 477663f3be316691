"""Chunked prefill against a KV cache (K1 + K2 reading the cache) on the GPU,
against the fp64 oracle, via the C ABI."""
import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import binding, inputs
from gpu_util import assert_close_attention, assert_within_one_ulp

pytestmark = pytest.mark.gpu


def chunk_inputs(B, Tq, Hq, Hkv, S_max, start_pos, seed):
    """A chunk of Tq tokens per sequence and caches holding start_pos[b]
    earlier rows (random bf16) with NaN poison from row start_pos[b] on."""
    x = inputs.prefill_inputs(B, Tq, Hq, Hkv, seed=seed)
    c = inputs.decode_inputs(B, Hq, Hkv, S_max, 0, 1, seed=seed + 1, start_pos=start_pos)
    x.update(k_cache=c["k_cache"], v_cache=c["v_cache"], start_pos=c["start_pos"])
    return x


def run_chunk(x, theta=1e6, eps=1e-6):
    d = {k: (t.cuda() if k != "start_pos" else t) for k, t in x.items()}
    out = binding.prefill_chunk(d["q"], d["k"], d["v"], d["k_cache"], d["v_cache"],
                                d["start_pos"], d["q_gamma"], d["k_gamma"], theta, eps)
    torch.cuda.synchronize()
    return out, d


def check_caches(x, d, k_rows, Tq):
    """Rows start_pos..start_pos+Tq-1 hold the chunk; every other row is as it was."""
    kc, vc = d["k_cache"].cpu(), d["v_cache"].cpu()
    for b, p in enumerate(x["start_pos"].tolist()):
        assert_within_one_ulp(kc[b, :, p:p + Tq].transpose(0, 1), k_rows[b], "appended keys")
        assert torch.equal(vc[b, :, p:p + Tq], x["v"][b].transpose(0, 1))
        assert torch.equal(kc[b, :, :p], x["k_cache"][b, :, :p])
        assert torch.equal(vc[b, :, :p], x["v_cache"][b, :, :p])
        assert torch.isnan(kc[b, :, p + Tq:].float()).all()
        assert torch.isnan(vc[b, :, p + Tq:].float()).all()


@pytest.mark.parametrize("Tq,Hq,Hkv,start_pos", [
    (1, 16, 8, [0, 5, 300]),            # one token: what decode computes
    (7, 32, 8, [0, 1, 127]),            # g = 4, a tile boundary in the cache
    (129, 8, 8, [0, 128, 1000]),        # g = 1, two Q tiles of the chunk
    (200, 16, 2, [3, 250, 0]),          # g = 8, ragged tails everywhere
    (64, 16, 1, [1024, 17, 511]),       # g = 16
])
def test_chunk_matches_oracle_and_fills_caches(cuda_lib, Tq, Hq, Hkv, start_pos):
    B, S = len(start_pos), 1400
    x = chunk_inputs(B, Tq, Hq, Hkv, S, start_pos, seed=Tq * 10 + Hq)
    ref, k_rows = oracle.prefill_chunk(x["q"], x["k"], x["v"], x["k_cache"], x["v_cache"],
                                       x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    out, d = run_chunk(x)
    assert_close_attention(out, ref, f"chunk Tq{Tq} Hq{Hq} Hkv{Hkv} start_pos {start_pos}")
    check_caches(x, d, k_rows, Tq)


def test_chunk_cache_ends_exactly_at_s_max(cuda_lib):
    """start_pos + Tq == S_max: the last key tile runs past the cache's end."""
    Tq, S = 100, 300
    x = chunk_inputs(2, Tq, 16, 4, S, [200, 0], seed=31)
    ref, k_rows = oracle.prefill_chunk(x["q"], x["k"], x["v"], x["k_cache"], x["v_cache"],
                                       x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    out, d = run_chunk(x)
    assert_close_attention(out, ref, "chunk at S_max")
    check_caches(x, d, k_rows, Tq)


def test_chunk_at_position_zero_is_prefill(cuda_lib):
    """With every start_pos = 0 a chunk is a plain prefill that also fills
    the caches: both outputs match the oracle's prefill (the chunk takes its
    query rows from the prologue, the plain prefill normalises them inside the
    attention kernel, so the two may differ in the last bit), and the cache
    holds what q3a_qknorm_rope writes for K."""
    B, T, Hq, Hkv, S = 2, 333, 32, 8, 512
    x = chunk_inputs(B, T, Hq, Hkv, S, [0, 0], seed=41)
    out, d = run_chunk(x)
    full = binding.prefill(d["q"], d["k"], d["v"], d["q_gamma"], d["k_gamma"], 1e6, 1e-6)
    khat = binding.qknorm_rope(d["k"], d["k_gamma"], 1e6, 1e-6)
    torch.cuda.synchronize()
    ref = oracle.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    assert_close_attention(out, ref, "chunk at position 0")
    assert_close_attention(full, ref, "prefill")
    assert float((out.float() - full.float()).abs().max()) <= 2e-2
    assert torch.equal(d["k_cache"][:, :, :T], khat.transpose(1, 2))
    assert torch.equal(d["v_cache"][:, :, :T], d["v"].transpose(1, 2))


def test_chunk_of_one_token_matches_decode(cuda_lib):
    """Tq = 1 computes what q3a_decode computes (two different kernels):
    both close to the oracle, and both append the same key row."""
    start_pos = [0, 63, 64, 999]
    B, Hq, Hkv, S = len(start_pos), 32, 8, 1000
    c = inputs.decode_inputs(B, Hq, Hkv, S, 0, 1, seed=51, start_pos=start_pos)
    dc = {k: (t.cuda() if k != "start_pos" else t) for k, t in c.items()}
    kc2, vc2 = dc["k_cache"].clone(), dc["v_cache"].clone()
    dec = binding.decode(dc["q"], dc["k_new"], dc["v_new"], dc["k_cache"], dc["v_cache"],
                         dc["start_pos"], dc["q_gamma"], dc["k_gamma"], 1e6, 1e-6)
    chk = binding.prefill_chunk(dc["q"][:, None].contiguous(), dc["k_new"][:, None].contiguous(),
                                dc["v_new"][:, None].contiguous(), kc2, vc2, dc["start_pos"],
                                dc["q_gamma"], dc["k_gamma"], 1e6, 1e-6)
    torch.cuda.synchronize()
    ref, _ = oracle.decode(c["q"], c["k_new"], c["v_new"], c["k_cache"], c["v_cache"],
                           c["start_pos"], c["q_gamma"], c["k_gamma"], 1e6, 1e-6)
    assert_close_attention(chk[:, 0], ref, "chunk Tq=1")
    assert_close_attention(dec, ref, "decode")
    assert torch.equal(kc2.view(torch.int16), dc["k_cache"].view(torch.int16))
    assert torch.equal(vc2.view(torch.int16), dc["v_cache"].view(torch.int16))


@pytest.mark.parametrize("T,cuts", [(6, [0, 2, 5, 6]), (700, [0, 300, 555, 700]),
                                    (520, [0, 1, 128, 129, 520])])
def test_chunks_in_sequence_equal_one_prefill(cuda_lib, T, cuts):
    """Feeding a sequence in chunks (the pages' [0:2], [2:5], [5:6] check, and
    longer ones across tile boundaries) gives the rows of one full prefill
    and leaves the caches holding every key and value."""
    B, Hq, Hkv, S = 2, 16, 4, 768
    xc = inputs.prefill_inputs(B, T, Hq, Hkv, seed=61 + T)
    ref = oracle.prefill(xc["q"], xc["k"], xc["v"], xc["q_gamma"], xc["k_gamma"], 1e6, 1e-6)
    x = {k: t.cuda() for k, t in xc.items()}
    full = binding.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    khat = binding.qknorm_rope(x["k"], x["k_gamma"], 1e6, 1e-6)
    kc = torch.full((B, Hkv, S, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sl = lambda t: t[:, a:b].contiguous()  # noqa: E731
        parts.append(binding.prefill_chunk(sl(x["q"]), sl(x["k"]), sl(x["v"]), kc, vc, [a] * B,
                                           x["q_gamma"], x["k_gamma"], 1e6, 1e-6))
    torch.cuda.synchronize()
    got = torch.cat(parts, 1)
    assert_close_attention(got, ref, f"chunks {cuts}")
    assert_close_attention(got, full.cpu().double(), f"chunks {cuts} against one prefill")
    assert torch.equal(kc[:, :, :T], khat.transpose(1, 2))
    assert torch.equal(vc[:, :, :T], x["v"].transpose(1, 2))
    assert torch.isnan(kc[:, :, T:].float()).all()


@pytest.mark.parametrize("gmax", [1.0, 2.3])
def test_chunk_large_gamma(cuda_lib, gmax):
    x = chunk_inputs(2, 150, 16, 4, 600, [0, 321], seed=71)
    g = torch.Generator().manual_seed(72)
    x["q_gamma"] = (torch.rand(128, generator=g) * gmax).to(torch.bfloat16)
    x["k_gamma"] = (torch.rand(128, generator=g) * gmax).to(torch.bfloat16)
    ref, k_rows = oracle.prefill_chunk(x["q"], x["k"], x["v"], x["k_cache"], x["v_cache"],
                                       x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    out, d = run_chunk(x)
    assert_close_attention(out, ref, f"chunk gamma max {gmax}")
    check_caches(x, d, k_rows, 150)


def test_chunk_context_overflow_leaves_caches_untouched(cuda_lib):
    x = chunk_inputs(2, 10, 8, 2, 128, [5, 119], seed=81)
    d = {k: (t.cuda() if k != "start_pos" else t) for k, t in x.items()}
    k0, v0 = d["k_cache"].clone(), d["v_cache"].clone()
    out = torch.full_like(d["q"], 3.0)
    with pytest.raises(binding.Q3AError) as e:
        binding.prefill_chunk(d["q"], d["k"], d["v"], d["k_cache"], d["v_cache"],
                              d["start_pos"], d["q_gamma"], d["k_gamma"], 1e6, 1e-6, out=out)
    assert e.value.status == binding.Q3A_ERANGE
    torch.cuda.synchronize()
    assert torch.equal(d["k_cache"].view(torch.int16), k0.view(torch.int16))
    assert torch.equal(d["v_cache"].view(torch.int16), v0.view(torch.int16))
    assert bool((out == 3.0).all())


def test_chunk_no_device_error_word(cuda_lib):
    x = chunk_inputs(1, 40, 8, 2, 256, [100], seed=91)
    d = {k: (t.cuda() if k != "start_pos" else t) for k, t in x.items()}
    ws = torch.empty(binding.prefill_chunk_workspace_size(1, 40, 8, 2), dtype=torch.uint8,
                     device="cuda")
    binding.prefill_chunk(d["q"], d["k"], d["v"], d["k_cache"], d["v_cache"], d["start_pos"],
                          d["q_gamma"], d["k_gamma"], 1e6, 1e-6, workspace=ws)
    assert binding.last_device_error(ws) == binding.Q3A_OK


@pytest.mark.slow
def test_chunk_qwen3_8b_shape(cuda_lib):
    """Qwen3-8B heads: four sequences, a 1024-token chunk each after 0, 1024,
    2047 and 3000 cached tokens in a 4096-row cache; the whole output and every
    appended row against the oracle."""
    start_pos = [0, 1024, 2047, 3000]
    B, Tq, Hq, Hkv, S = 4, 1024, 32, 8, 4096
    x = chunk_inputs(B, Tq, Hq, Hkv, S, start_pos, seed=101)
    out, d = run_chunk(x)
    ref, k_rows = oracle.prefill_chunk(x["q"], x["k"], x["v"], x["k_cache"], x["v_cache"],
                                       x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    assert_close_attention(out, ref, "chunk qwen3-8b")
    check_caches(x, d, k_rows, Tq)


def test_chunk_more_items_than_ctas_with_tails(cuda_lib):
    """160 work items (five pairs of 32-token Q tiles for each of 32 (b, kv)
    groups) on persistent CTAs, so several CTAs take more than one item, and
    every sequence's valid keys end inside a 128-key tile (a NaN-poisoned V
    tail to clear per item). Every output row against the oracle."""
    B, Tq, Hq, Hkv, S = 4, 300, 32, 8, 2400
    x = chunk_inputs(B, Tq, Hq, Hkv, S, [100, 1000, 1501, 1999], seed=33)
    out, d = run_chunk(x)
    ref, k_rows = oracle.prefill_chunk(x["q"], x["k"], x["v"], x["k_cache"], x["v_cache"],
                                       x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    assert bool(torch.isfinite(out).all())
    assert_close_attention(out, ref, "160 chunk items with tails")
    check_caches(x, d, k_rows, Tq)


@pytest.mark.parametrize("scale,expect_error", [(1.5, False), (1.0e4, True)])
def test_chunk_cache_above_the_bound(cuda_lib, scale, expect_error):
    """The chunk's softmax shift comes from the norm bound of keys written by
    this library. Cached keys 1.5 times too long break the bound, but the shift
    cancels: the output still matches the oracle. Keys 10^4 times too long
    overflow the softmax sum: the call reports Q3A_EINVAL through the error
    word instead of returning silent NaN."""
    B, Tq, Hq, Hkv, S = 2, 40, 16, 4, 600
    x = chunk_inputs(B, Tq, Hq, Hkv, S, [300, 450], seed=35)
    for b, p in enumerate([300, 450]):
        x["k_cache"][b, :, :p] = (x["k_cache"][b, :, :p].float() * scale).to(torch.bfloat16)
    d = {k: (t.cuda() if k != "start_pos" else t) for k, t in x.items()}
    ws = torch.empty(binding.prefill_chunk_workspace_size(B, Tq, Hq, Hkv), dtype=torch.uint8,
                     device="cuda")
    out = binding.prefill_chunk(d["q"], d["k"], d["v"], d["k_cache"], d["v_cache"],
                                d["start_pos"], d["q_gamma"], d["k_gamma"], 1e6, 1e-6,
                                workspace=ws)
    torch.cuda.synchronize()
    status = binding.last_device_error(ws)
    if expect_error:
        assert status == binding.Q3A_EINVAL
    else:
        assert status == binding.Q3A_OK
        ref, _ = oracle.prefill_chunk(x["q"], x["k"], x["v"], x["k_cache"], x["v_cache"],
                                      x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
        assert_close_attention(out, ref, "cache keys x1.5")
