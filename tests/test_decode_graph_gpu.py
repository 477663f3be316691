"""Decode with device-resident positions (q3a_decode_device_pos): the same
bits as the host-position decode, the device-side range check, and replays
of a captured CUDA graph that advances the positions on the device."""
import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import binding, inputs
from gpu_util import assert_close_attention

pytestmark = pytest.mark.gpu


def to_dev(x):
    return {k: (t.cuda() if k != "start_pos" else t) for k, t in x.items()}


@pytest.mark.parametrize("Hq,Hkv,start_pos", [(32, 8, [0, 1, 1023, 1024, 2999]),
                                              (16, 1, [5, 700]), (8, 8, [2047])])
def test_device_positions_match_host_positions(cuda_lib, Hq, Hkv, start_pos):
    B, S = len(start_pos), 3000
    x = inputs.decode_inputs(B, Hq, Hkv, S, 0, 1, seed=Hq + 3 * Hkv, start_pos=start_pos)
    a, b = to_dev(x), to_dev(x)
    a["k_cache"], a["v_cache"] = a["k_cache"].clone(), a["v_cache"].clone()
    host = binding.decode(a["q"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"],
                          x["start_pos"], a["q_gamma"], a["k_gamma"], 1e6, 1e-6)
    ws = torch.empty(binding.decode_workspace_size(B, Hq, Hkv, S), dtype=torch.uint8,
                     device="cuda")
    dev = binding.decode_device_pos(b["q"], b["k_new"], b["v_new"], b["k_cache"], b["v_cache"],
                                    x["start_pos"].cuda(), b["q_gamma"], b["k_gamma"], 1e6, 1e-6,
                                    workspace=ws)
    torch.cuda.synchronize()
    assert binding.last_device_error(ws) == binding.Q3A_OK
    assert torch.equal(host, dev)
    assert torch.equal(a["k_cache"].view(torch.int16), b["k_cache"].view(torch.int16))
    assert torch.equal(a["v_cache"].view(torch.int16), b["v_cache"].view(torch.int16))
    ref, _ = oracle.decode(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                           x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    assert_close_attention(dev, ref, "device positions")


@pytest.mark.parametrize("bad", [[5, 128], [-1, 3], [0, 1 << 20]])
def test_device_range_check_writes_nothing(cuda_lib, bad):
    B, Hq, Hkv, S = 2, 8, 2, 128
    x = to_dev(inputs.decode_inputs(B, Hq, Hkv, S, 0, 1, seed=7, start_pos=[3, 4]))
    k0, v0 = x["k_cache"].clone(), x["v_cache"].clone()
    out = torch.full_like(x["q"], 3.0)
    ws = torch.empty(binding.decode_workspace_size(B, Hq, Hkv, S), dtype=torch.uint8,
                     device="cuda")
    pos = torch.tensor(bad, dtype=torch.int32, device="cuda")
    binding.decode_device_pos(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], pos,
                              x["q_gamma"], x["k_gamma"], 1e6, 1e-6, out=out, workspace=ws)
    assert binding.last_device_error(ws) == binding.Q3A_ERANGE
    assert torch.equal(x["k_cache"].view(torch.int16), k0.view(torch.int16))
    assert torch.equal(x["v_cache"].view(torch.int16), v0.view(torch.int16))
    assert bool((out == 3.0).all())
    # the same workspace serves a valid call afterwards
    pos.copy_(torch.tensor([3, 4], dtype=torch.int32))
    binding.decode_device_pos(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"], pos,
                              x["q_gamma"], x["k_gamma"], 1e6, 1e-6, out=out, workspace=ws)
    assert binding.last_device_error(ws) == binding.Q3A_OK
    assert not bool((out == 3.0).all())


def test_graph_replays_equal_eager_steps(cuda_lib):
    """A decode step and the position increment captured once in a CUDA graph,
    replayed for several tokens, gives the bits of the same steps run eagerly
    with host positions."""
    B, Hq, Hkv, S, steps = 3, 32, 8, 2048, 6
    start = [0, 700, 1500]
    x = inputs.decode_inputs(B, Hq, Hkv, S, 0, 1, seed=11, start_pos=start)
    g = torch.Generator().manual_seed(12)
    new = [{k: (torch.randn(x[k].shape, generator=g)).to(torch.bfloat16).cuda()
            for k in ("q", "k_new", "v_new")} for _ in range(steps)]
    gam = {k: x[k].cuda() for k in ("q_gamma", "k_gamma")}
    # eager, host positions
    kc_e, vc_e = x["k_cache"].cuda(), x["v_cache"].cuda()
    eager = []
    for s in range(steps):
        eager.append(binding.decode(new[s]["q"], new[s]["k_new"], new[s]["v_new"], kc_e, vc_e,
                                    [p + s for p in start], gam["q_gamma"], gam["k_gamma"],
                                    1e6, 1e-6).clone())
    # captured graph, device positions
    kc_g, vc_g = x["k_cache"].cuda(), x["v_cache"].cuda()
    bufs = {k: torch.empty_like(new[0][k]) for k in ("q", "k_new", "v_new")}
    out = torch.empty_like(bufs["q"])
    pos = torch.tensor(start, dtype=torch.int32, device="cuda")
    ws = torch.empty(binding.decode_workspace_size(B, Hq, Hkv, S), dtype=torch.uint8,
                     device="cuda")
    for k in bufs:
        bufs[k].copy_(new[0][k])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.decode_device_pos(bufs["q"], bufs["k_new"], bufs["v_new"], kc_g, vc_g, pos,
                                  gam["q_gamma"], gam["k_gamma"], 1e6, 1e-6, out=out,
                                  workspace=ws)
        pos.add_(1)
    torch.cuda.synchronize()
    # capture does not run the work: caches, positions and out are unchanged
    assert torch.equal(pos.cpu(), torch.tensor(start, dtype=torch.int32))
    for s in range(steps):
        for k in bufs:
            bufs[k].copy_(new[s][k])
        graph.replay()
        torch.cuda.synchronize()
        assert binding.last_device_error(ws) == binding.Q3A_OK
        assert torch.equal(out, eager[s]), f"step {s}"
    assert torch.equal(kc_g.view(torch.int16), kc_e.view(torch.int16))
    assert torch.equal(vc_g.view(torch.int16), vc_e.view(torch.int16))
    assert torch.equal(pos.cpu(), torch.tensor([p + steps for p in start], dtype=torch.int32))
