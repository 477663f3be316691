"""Gated decode (Qwen3-Next / Qwen3.5 global layer, head_dim 256) on the GPU
against the fp64 oracle, via the C ABI: outputs, the appended cache rows, and
a full-size workload on sampled sequences."""
import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import binding, inputs
from gpu_util import assert_close_attention, assert_within_one_ulp

pytestmark = pytest.mark.gpu


def to_dev(x):
    return {k: (t.cuda() if k != "start_pos" else t) for k, t in x.items()}


@pytest.mark.parametrize("Hq,Hkv,d_r,start_pos", [
    (16, 2, 64, [0, 1, 1023, 1024, 2047]),   # Qwen3-Next heads; split boundaries
    (8, 2, 64, [5, 700, 1500]),              # Qwen3.5-0.8B heads
    (32, 2, 64, [2999, 64]),                 # g = 16
    (4, 4, 256, [300]),                      # g = 1, full rotary
    (8, 4, 0, [17, 1100]),                   # no rotary
    (24, 4, 64, [900, 2500]),                # g = 6 (Qwen3.5-27B heads)
    (24, 2, 64, [3, 2100]),                  # g = 12
])
def test_gated_decode_matches_oracle_and_appends(cuda_lib, Hq, Hkv, d_r, start_pos):
    B, S = len(start_pos), 3000
    x = inputs.gated_decode_inputs(B, Hq, Hkv, S, 0, 1, seed=Hq + 5 * Hkv + d_r,
                                   start_pos=start_pos)
    d = to_dev(x)
    out = binding.gated_decode(d["qg"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                               x["start_pos"], d["q_w"], d["k_w"], d_r, 1e7, 1e-6)
    torch.cuda.synchronize()
    ref, k_row = oracle.gated_decode(x["qg"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                                     x["start_pos"], x["q_w"], x["k_w"], d_r, 1e7, 1e-6)
    assert_close_attention(out, ref, f"gated decode Hq{Hq} Hkv{Hkv} d_r{d_r}")
    kc, vc = d["k_cache"].cpu(), d["v_cache"].cpu()
    for b, p in enumerate(start_pos):
        assert_within_one_ulp(kc[b, :, p], k_row[b], f"appended key b{b}")
        assert torch.equal(vc[b, :, p].view(torch.int16), x["v_new"][b].view(torch.int16))
        # rows before p untouched, rows after p still NaN
        assert torch.equal(kc[b, :, :p].view(torch.int16), x["k_cache"][b, :, :p].view(torch.int16))
        assert bool(torch.isnan(kc[b, :, p + 1:].float()).all())


def test_gated_decode_steps_extend_a_prefill(cuda_lib):
    """Four decode steps after a 200-token prompt whose keys went into the cache
    through the oracle: each step's output matches the oracle's prefill row of
    the grown sequence (to the cache's bf16 rounding)."""
    T0, steps, Hq, Hkv, D = 200, 4, 16, 2, 256
    x = inputs.gated_inputs(1, T0 + steps, Hq, Hkv, seed=12)
    full = oracle.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], 64, 1e7, 1e-6)
    khat = oracle.gated_qknorm_rope(x["k"], x["k_w"], D, 64, 1e7, 1e-6).to(torch.bfloat16)
    S = T0 + steps + 8
    kc = torch.full((1, Hkv, S, D), float("nan"), dtype=torch.bfloat16)
    vc = torch.full_like(kc, float("nan"))
    kc[0, :, :T0] = khat[0, :T0].transpose(0, 1)
    vc[0, :, :T0] = x["v"][0, :T0].transpose(0, 1)
    kc, vc = kc.cuda(), vc.cuda()
    qw, kw = x["q_w"].cuda(), x["k_w"].cuda()
    for s in range(steps):
        t = T0 + s
        out = binding.gated_decode(x["qg"][:, t].contiguous().cuda(), x["k"][:, t].contiguous().cuda(),
                                   x["v"][:, t].contiguous().cuda(), kc, vc, [t], qw, kw, 64, 1e7,
                                   1e-6)
        torch.cuda.synchronize()
        assert_close_attention(out[0], full[0, t], f"step {s}")


def test_gated_decode_device_positions_and_graph_replay(cuda_lib):
    """Device-resident positions give the bits of host positions; a captured
    graph of the step plus the position increment, replayed, equals eager
    steps; an out-of-range position writes nothing and reports ERANGE."""
    B, Hq, Hkv, S, steps = 2, 16, 2, 2048, 4
    start = [10, 1500]
    x = inputs.gated_decode_inputs(B, Hq, Hkv, S, 0, 1, seed=13, start_pos=start)
    g = torch.Generator().manual_seed(14)
    new = [{k: torch.randn(x[k].shape, generator=g).to(torch.bfloat16).cuda()
            for k in ("qg", "k_new", "v_new")} for _ in range(steps)]
    qw, kw = x["q_w"].cuda(), x["k_w"].cuda()
    kc_e, vc_e = x["k_cache"].cuda(), x["v_cache"].cuda()
    eager = [binding.gated_decode(new[s]["qg"], new[s]["k_new"], new[s]["v_new"], kc_e, vc_e,
                                  [p + s for p in start], qw, kw, 64, 1e7, 1e-6).clone()
             for s in range(steps)]
    kc_g, vc_g = x["k_cache"].cuda(), x["v_cache"].cuda()
    bufs = {k: torch.empty_like(new[0][k]) for k in ("qg", "k_new", "v_new")}
    out = torch.empty((B, Hq, 256), dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor(start, dtype=torch.int32, device="cuda")
    ws = torch.empty(binding.gated_decode_workspace_size(B, Hq, Hkv, S), dtype=torch.uint8,
                     device="cuda")
    for k in bufs:
        bufs[k].copy_(new[0][k])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.gated_decode_device_pos(bufs["qg"], bufs["k_new"], bufs["v_new"], kc_g, vc_g,
                                        pos, qw, kw, 64, 1e7, 1e-6, out=out, workspace=ws)
        pos.add_(1)
    torch.cuda.synchronize()
    for s in range(steps):
        for k in bufs:
            bufs[k].copy_(new[s][k])
        graph.replay()
        torch.cuda.synchronize()
        assert binding.last_device_error(ws) == binding.Q3A_OK
        assert torch.equal(out, eager[s]), f"step {s}"
    assert torch.equal(kc_g.view(torch.int16), kc_e.view(torch.int16))
    assert torch.equal(vc_g.view(torch.int16), vc_e.view(torch.int16))
    # out of range: nothing written
    k0 = kc_g.clone()
    out.fill_(3.0)
    bad = torch.tensor([5, S], dtype=torch.int32, device="cuda")
    binding.gated_decode_device_pos(bufs["qg"], bufs["k_new"], bufs["v_new"], kc_g, vc_g, bad,
                                    qw, kw, 64, 1e7, 1e-6, out=out, workspace=ws)
    assert binding.last_device_error(ws) == binding.Q3A_ERANGE
    assert torch.equal(kc_g.view(torch.int16), k0.view(torch.int16))
    assert bool((out == 3.0).all())
