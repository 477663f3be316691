"""q3a_decode_noalloc: the decode step for callers that cannot allocate device
memory (its scratch is a fixed static device array inside the library).

Checked through the C ABI against q3a_decode, the entry point that takes a
caller workspace, on two calls in a row (the second call runs on the array the
first one left behind), plus the size limit. This file is collected last.
"""
import ctypes

import pytest
import torch

from qwen3_qk_norm_gb300 import binding, inputs
from gpu_util import assert_close_attention

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 * 1024 * 1024  # Q3A_DECODE_NOALLOC_SCRATCH_BYTES in include/q3a.h


def _dev(x):
    return {k: (t.cuda() if k != "start_pos" else t) for k, t in x.items()}


def _noalloc(lib, d, k_cache, v_cache, out, Hq, Hkv, S_max):
    B = d["q"].shape[0]
    sp = d["start_pos"].to(torch.int32).contiguous()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.q3a_decode_noalloc(d["q"].data_ptr(), d["k_new"].data_ptr(), d["v_new"].data_ptr(),
                                  k_cache.data_ptr(), v_cache.data_ptr(), sp.data_ptr(),
                                  d["q_gamma"].data_ptr(), d["k_gamma"].data_ptr(),
                                  out.data_ptr(), B, Hq, Hkv, 128, S_max, 1e6, 1e-6, stream)


@pytest.mark.parametrize("cases", [[(41, 32, 8, [5, 1500, 2999, 0]),
                                    (42, 32, 4, [2047, 10, 700, 1024, 64])]])
def test_decode_noalloc_matches_decode_on_two_calls_in_a_row(cuda_lib, cases):
    lib = binding.load()
    S_max = 3000
    for seed, Hq, Hkv, sp in cases:
        x = inputs.decode_inputs(len(sp), Hq, Hkv, S_max, 0, 1, seed=seed, start_pos=sp)
        d = _dev(x)
        kc_ref, vc_ref = d["k_cache"].clone(), d["v_cache"].clone()
        ref = binding.decode(d["q"], d["k_new"], d["v_new"], kc_ref, vc_ref, d["start_pos"],
                             d["q_gamma"], d["k_gamma"], 1e6, 1e-6)
        kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
        out = torch.full_like(d["q"], float("nan"))
        assert _noalloc(lib, d, kc, vc, out, Hq, Hkv, S_max) == binding.Q3A_OK
        torch.cuda.synchronize()
        assert_close_attention(out, ref.double().cpu(), f"noalloc vs decode, seed {seed}")
        # the cache append is the same as q3a_decode's
        assert torch.equal(kc.view(torch.int16), kc_ref.view(torch.int16))
        assert torch.equal(vc.view(torch.int16), vc_ref.view(torch.int16))


def test_decode_noalloc_rejects_calls_beyond_its_scratch(cuda_lib):
    lib = binding.load()
    # batch 64 x 8 groups x 4 heads x 32 splits of 520 bytes = 34 MB > 16 MiB
    B, Hq, Hkv, S_max = 64, 32, 8, 32768
    need = 256 + 4 * 130 * B * Hkv * (Hq // Hkv) * 32
    assert need > SCRATCH_BYTES
    q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((B, Hkv, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(128, dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((1, 128), dtype=torch.bfloat16, device="cuda")  # never touched
    out = torch.full_like(q, 5.0)
    sp = torch.full((B,), S_max - 1, dtype=torch.int32)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.q3a_decode_noalloc(q.data_ptr(), kn.data_ptr(), kn.data_ptr(), cache.data_ptr(),
                                cache.data_ptr(), sp.data_ptr(), g.data_ptr(), g.data_ptr(),
                                out.data_ptr(), B, Hq, Hkv, 128, S_max, 1e6, 1e-6, stream)
    assert st == binding.Q3A_EINVAL
    torch.cuda.synchronize()
    assert bool((out == 5.0).all())
