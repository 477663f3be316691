"""q3a_decode_noalloc: the decode step for callers that cannot allocate device
memory (a plugin whose host framework owns every device allocation, or a
serving loop that must not call cudaMalloc because it can synchronise the
device). Its scratch is a fixed static device array inside the library.

Checked through the C ABI against q3a_decode, the entry point that takes a
caller workspace and runs the same kernels: the outputs and the cache appends
must be bit-identical, on two calls in a row (the second call runs on the
array the first one left behind), and one call is also compared with the fp64
oracle. Also: the calls leave the device's free memory unchanged, the error
word is readable, and the size limit holds at its exact boundary. This file is
collected last.
"""
import ctypes

import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import binding, inputs
from gpu_util import assert_close_attention

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 * 1024 * 1024  # Q3A_DECODE_NOALLOC_SCRATCH_BYTES in include/q3a.h
SPLIT_KEYS = 1024                  # keys per split of the head_dim-128 decode
PARTIAL_BYTES = 4 * 130            # m, l and acc[128] in fp32 per (split, head)


def _need(B, Hq, max_pos):
    return 256 + PARTIAL_BYTES * B * Hq * ((max_pos + 1 + SPLIT_KEYS - 1) // SPLIT_KEYS)


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
    for i, (seed, Hq, Hkv, sp) in enumerate(cases):
        x = inputs.decode_inputs(len(sp), Hq, Hkv, S_max, 0, 1, seed=seed, start_pos=sp)
        d = _dev(x)
        kc_ref, vc_ref = d["k_cache"].clone(), d["v_cache"].clone()
        ref = binding.decode(d["q"], d["k_new"], d["v_new"], kc_ref, vc_ref, d["start_pos"],
                             d["q_gamma"], d["k_gamma"], 1e6, 1e-6)
        kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
        out = torch.full_like(d["q"], float("nan"))
        assert _noalloc(lib, d, kc, vc, out, Hq, Hkv, S_max) == binding.Q3A_OK
        torch.cuda.synchronize()
        assert binding.last_device_error(None) == binding.Q3A_OK
        # same kernels, same inputs: the same bits as q3a_decode
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"seed {seed}"
        assert torch.equal(kc.view(torch.int16), kc_ref.view(torch.int16))
        assert torch.equal(vc.view(torch.int16), vc_ref.view(torch.int16))
        if i == 0:  # and within the attention tolerance of the fp64 oracle
            want, _ = oracle.decode(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                                    x["start_pos"], x["q_gamma"], x["k_gamma"], 1e6, 1e-6)
            assert_close_attention(out, want, f"noalloc vs oracle, seed {seed}")


def test_decode_noalloc_allocates_nothing(cuda_lib):
    """After a warm-up call (which loads the library's device code), further
    calls change neither the device's free memory nor torch's allocations."""
    lib = binding.load()
    S_max, Hq, Hkv, sp = 2100, 16, 4, [2099, 3, 1024]
    d = _dev(inputs.decode_inputs(len(sp), Hq, Hkv, S_max, 0, 1, seed=43, start_pos=sp))
    out = torch.empty_like(d["q"])
    assert _noalloc(lib, d, d["k_cache"], d["v_cache"], out, Hq, Hkv, S_max) == binding.Q3A_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(5):
        assert _noalloc(lib, d, d["k_cache"], d["v_cache"], out, Hq, Hkv, S_max) == binding.Q3A_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0
    assert binding.last_device_error(None) == binding.Q3A_OK


def test_decode_noalloc_size_limit_at_its_exact_boundary(cuda_lib):
    """The largest call that fits: 77 sequences x 1 head x 419 splits =
    32263 partials, 256 + 520 * 32263 = 16777016 bytes (200 under 16 MiB); it
    runs and gives q3a_decode's bits. One partial more (109 sequences x 296
    splits = 32264, 16777536 bytes) is rejected before anything is written."""
    lib = binding.load()
    # fits: one long sequence sets the split count, the others are short
    B, S_max = 77, 419 * SPLIT_KEYS
    sp = [S_max - 1] + [b % 50 for b in range(1, B)]
    assert _need(B, 1, max(sp)) == 16777016 <= SCRATCH_BYTES
    g = torch.Generator(device="cuda").manual_seed(44)
    kc = torch.zeros((B, 1, S_max, 128), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    vc[0, 0, : S_max - 1].normal_(generator=g)
    kc[0, 0, : S_max - 1].normal_(generator=g)
    x = inputs.decode_inputs(B, 1, 1, 8, 0, 1, seed=45, start_pos=[0] * B)
    d = _dev({k: x[k] for k in ("q", "k_new", "v_new", "q_gamma", "k_gamma")})
    d["start_pos"] = torch.tensor(sp, dtype=torch.int32)
    ref = binding.decode(d["q"], d["k_new"], d["v_new"], kc, vc, d["start_pos"], d["q_gamma"],
                         d["k_gamma"], 1e6, 1e-6)
    out = torch.full_like(d["q"], float("nan"))
    # the decode above appended the same rows that this call appends again
    assert _noalloc(lib, d, kc, vc, out, 1, 1, S_max) == binding.Q3A_OK
    torch.cuda.synchronize()
    assert binding.last_device_error(None) == binding.Q3A_OK
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    del kc, vc
    # one partial over: rejected, nothing written (the caches are never read)
    B, S_max = 109, 296 * SPLIT_KEYS
    sp = torch.zeros(B, dtype=torch.int32)
    sp[5] = S_max - 1
    assert _need(B, 1, S_max - 1) == 16777536 > SCRATCH_BYTES
    q = torch.zeros((B, 1, 128), dtype=torch.bfloat16, device="cuda")
    gam = torch.ones(128, dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((1, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, 5.0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.q3a_decode_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), cache.data_ptr(),
                                cache.data_ptr(), sp.data_ptr(), gam.data_ptr(), gam.data_ptr(),
                                out.data_ptr(), B, 1, 1, 128, S_max, 1e6, 1e-6, stream)
    assert st == binding.Q3A_EINVAL
    torch.cuda.synchronize()
    assert bool((out == 5.0).all())


def test_decode_noalloc_rejects_calls_beyond_its_scratch(cuda_lib):
    lib = binding.load()
    # batch 64 x 8 groups x 4 heads x 32 splits of 520 bytes = 34 MB > 16 MiB
    B, Hq, Hkv, S_max = 64, 32, 8, 32768
    need = _need(B, Hq, S_max - 1)
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
