"""Split-KV decode (K3 + K4) on the GPU against the fp64 oracle, via the C ABI."""
import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import binding, inputs
from gpu_util import assert_close_attention, assert_within_one_ulp

pytestmark = pytest.mark.gpu


def run_decode(x, theta=1e6, eps=1e-6):
    d = {k: (t.cuda() if k != "start_pos" else t) for k, t in x.items()}
    out = binding.decode(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                         d["start_pos"], d["q_gamma"], d["k_gamma"], theta, eps)
    torch.cuda.synchronize()
    return out, d


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (32, 8), (32, 4), (32, 2)])
def test_decode_small_matches_oracle_and_appends(cuda_lib, Hq, Hkv):
    start_pos = [0, 1, 63, 64, 1023, 1024, 2500, 2999]
    B, S = len(start_pos), 3000
    x = inputs.decode_inputs(B, Hq, Hkv, S, 0, 1, seed=Hq + Hkv, start_pos=start_pos)
    ref, k_row = oracle.decode(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                               x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    out, d = run_decode(x)
    assert_close_attention(out, ref, f"decode Hq{Hq} Hkv{Hkv}")
    kc, vc = d["k_cache"].cpu(), d["v_cache"].cpu()
    for b, p in enumerate(start_pos):
        assert_within_one_ulp(kc[b, :, p], k_row[b], "appended key")
        assert torch.equal(vc[b, :, p], x["v_new"][b])
        # rows before p untouched, rows after p untouched (still NaN poison)
        assert torch.equal(kc[b, :, :p], x["k_cache"][b, :, :p])
        assert torch.equal(vc[b, :, :p], x["v_cache"][b, :, :p])
        assert torch.isnan(kc[b, :, p + 1:].float()).all()
        assert torch.isnan(vc[b, :, p + 1:].float()).all()


def test_decode_context_overflow_leaves_caches_untouched(cuda_lib):
    x = inputs.decode_inputs(2, 8, 2, 128, 0, 1, seed=3, start_pos=[5, 128])
    d = {k: (t.cuda() if k != "start_pos" else t) for k, t in x.items()}
    k0, v0 = d["k_cache"].clone(), d["v_cache"].clone()
    out = torch.full_like(d["q"], 3.0)
    with pytest.raises(binding.Q3AError) as e:
        binding.decode(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                       d["start_pos"], d["q_gamma"], d["k_gamma"], 1e6, 1e-6, out=out)
    assert e.value.status == binding.Q3A_ERANGE
    torch.cuda.synchronize()
    assert torch.equal(d["k_cache"].view(torch.int16), k0.view(torch.int16))
    assert torch.equal(d["v_cache"].view(torch.int16), v0.view(torch.int16))
    assert bool((out == 3.0).all())


def test_decode_of_last_token_equals_prefill_last_row(cuda_lib):
    """Prefill then decode (the chunked-cache check of the pages' §20.9): a
    cache filled with K1's normalised+rotated keys, decode at p = T-1."""
    T, Hq, Hkv, S = 777, 32, 8, 1024
    x = {k: t.cuda() for k, t in inputs.prefill_inputs(1, T, Hq, Hkv, seed=21).items()}
    full = binding.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    khat = binding.qknorm_rope(x["k"], x["k_gamma"], 1e6, 1e-6)
    k_cache = torch.full((1, Hkv, S, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    v_cache = torch.full_like(k_cache, float("nan"))
    k_cache[0, :, : T - 1] = khat[0, : T - 1].transpose(0, 1)
    v_cache[0, :, : T - 1] = x["v"][0, : T - 1].transpose(0, 1)
    out = binding.decode(x["q"][:, T - 1].contiguous(), x["k"][:, T - 1].contiguous(),
                         x["v"][:, T - 1].contiguous(), k_cache, v_cache, [T - 1],
                         x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
    torch.cuda.synchronize()
    diff = (out[0].float() - full[0, T - 1].float()).abs().max()
    assert float(diff) < 2e-2
    # the appended key row is K1's row T-1
    assert torch.equal(k_cache[0, :, T - 1], khat[0, T - 1])


def test_decode_no_device_error_word(cuda_lib):
    x = inputs.decode_inputs(2, 8, 2, 300, 0, 1, seed=4, start_pos=[10, 299])
    d = {k: (t.cuda() if k != "start_pos" else t) for k, t in x.items()}
    ws = torch.empty(binding.decode_workspace_size(2, 8, 2, 300), dtype=torch.uint8,
                     device="cuda")
    binding.decode(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["start_pos"],
                   d["q_gamma"], d["k_gamma"], 1e6, 1e-6, workspace=ws)
    assert binding.last_device_error(ws) == binding.Q3A_OK
