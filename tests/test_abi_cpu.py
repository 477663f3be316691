"""Host-side checks of the C ABI: the library loads, exports every function
include/q3a.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

from qwen3_qk_norm_gb300 import binding
from qwen3_qk_norm_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "q3a.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q3a_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert "q3a_prefill" in names and "q3a_decode" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(binding.EXPORTED) == names


def test_status_strings(lib):
    for s in range(6):
        assert lib.q3a_status_string(s)
    assert b"range" in lib.q3a_status_string(binding.Q3A_ERANGE)


FAKE = 1 << 20  # an aligned non-null address; never dereferenced on rejected calls


def prefill_call(lib, **kw):
    a = dict(B=1, T=4, Hq=32, Hkv=8, d=128, theta=1e6, eps=1e-6, ws=FAKE, ws_bytes=1 << 40)
    a.update(kw)
    return lib.q3a_prefill(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["B"], a["T"], a["Hq"], a["Hkv"],
                           a["d"], a["theta"], a["eps"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw", [dict(d=64), dict(d=256), dict(Hq=30), dict(Hq=96, Hkv=3),
                                dict(Hq=64, Hkv=2), dict(eps=0.0), dict(eps=-1.0),
                                dict(theta=1.0), dict(theta=float("nan")), dict(B=-1),
                                dict(T=-2), dict(ws=FAKE + 16), dict(ws=0), dict(ws_bytes=1024)])
def test_prefill_rejects_bad_arguments(lib, kw):
    assert prefill_call(lib, **kw) == binding.Q3A_EINVAL


def test_prefill_empty_shapes_launch_nothing(lib):
    assert prefill_call(lib, B=0) == binding.Q3A_OK
    assert prefill_call(lib, T=0) == binding.Q3A_OK


def test_prefill_null_or_misaligned_pointer(lib):
    args = [FAKE] * 6
    for i in range(6):
        for bad in (0, FAKE + 2):
            a = list(args)
            a[i] = bad
            st = lib.q3a_prefill(*a, 1, 4, 32, 8, 128, 1e6, 1e-6, FAKE, 1 << 40, None)
            assert st == binding.Q3A_EINVAL


def decode_call(lib, start_pos, S_max=64, **kw):
    B = len(start_pos)
    sp = (ctypes.c_int32 * B)(*start_pos)
    a = dict(Hq=32, Hkv=8, d=128, theta=1e6, eps=1e-6, ws=FAKE, ws_bytes=1 << 40)
    a.update(kw)
    return lib.q3a_decode(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.addressof(sp), FAKE, FAKE, FAKE, B,
                          a["Hq"], a["Hkv"], a["d"], S_max, a["theta"], a["eps"], a["ws"],
                          a["ws_bytes"], None)


@pytest.mark.parametrize("sp", [[64], [0, 64], [-1], [5, 100, 3]])
def test_decode_context_overflow_is_erange(lib, sp):
    """start_pos + 1 > S_max (or negative) is refused before anything is written."""
    assert decode_call(lib, sp, S_max=64) == binding.Q3A_ERANGE


def test_decode_rejects_bad_arguments(lib):
    assert decode_call(lib, [3], d=64) == binding.Q3A_EINVAL
    assert decode_call(lib, [3], Hq=12, Hkv=8) == binding.Q3A_EINVAL
    assert decode_call(lib, [3], ws_bytes=16) == binding.Q3A_EINVAL
    assert decode_call(lib, [3] * 2049) == binding.Q3A_EINVAL
    assert decode_call(lib, [], S_max=64) == binding.Q3A_OK


def test_workspace_sizes(lib):
    B, T, Hq, Hkv = 4, 4096, 32, 8
    ws = binding.prefill_workspace_size(B, T, Hq, Hkv)
    assert ws >= 256 + B * T * Hkv * 128 * 2  # header and the normalised keys
    assert binding.prefill_workspace_size(B, T, Hq, Hkv, 64) == 0
    dws = binding.decode_workspace_size(64, 32, 8, 32768)
    assert dws >= 256 + 64 * 8 * 32 * 4 * 130 * 4


def chunk_call(lib, start_pos, Tq=4, S_max=64, **kw):
    B = len(start_pos)
    sp = (ctypes.c_int32 * B)(*start_pos)
    a = dict(Hq=32, Hkv=8, d=128, theta=1e6, eps=1e-6, ws=FAKE, ws_bytes=1 << 40)
    a.update(kw)
    return lib.q3a_prefill_chunk(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.addressof(sp), FAKE, FAKE,
                                 FAKE, B, Tq, a["Hq"], a["Hkv"], a["d"], S_max, a["theta"],
                                 a["eps"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("sp,Tq", [([61], 4), ([0, 61], 4), ([-1], 1), ([0], 65), ([63], 2)])
def test_chunk_context_overflow_is_erange(lib, sp, Tq):
    """start_pos + Tq > S_max (or a negative position) is refused before any write."""
    assert chunk_call(lib, sp, Tq=Tq, S_max=64) == binding.Q3A_ERANGE


def test_chunk_rejects_bad_arguments(lib):
    assert chunk_call(lib, [3], d=64) == binding.Q3A_EINVAL
    assert chunk_call(lib, [3], Hq=12, Hkv=8) == binding.Q3A_EINVAL
    assert chunk_call(lib, [3], ws_bytes=16) == binding.Q3A_EINVAL
    assert chunk_call(lib, [3], ws=FAKE + 16) == binding.Q3A_EINVAL
    assert chunk_call(lib, [3], S_max=0) == binding.Q3A_EINVAL
    assert chunk_call(lib, [3] * 2049, S_max=64) == binding.Q3A_EINVAL
    assert chunk_call(lib, [3], Hq=256, Hkv=256) == binding.Q3A_EINVAL  # Hq + 2 Hkv > 512
    assert chunk_call(lib, [], S_max=64) == binding.Q3A_OK
    assert chunk_call(lib, [3], Tq=0) == binding.Q3A_OK


def test_chunk_null_or_misaligned_pointer(lib):
    sp = (ctypes.c_int32 * 1)(3)
    args = [FAKE] * 9
    args[5] = ctypes.addressof(sp)
    for i in [0, 1, 2, 3, 4, 6, 7, 8]:
        for bad in (0, FAKE + 2):
            a = list(args)
            a[i] = bad
            st = lib.q3a_prefill_chunk(*a, 1, 4, 32, 8, 128, 64, 1e6, 1e-6, FAKE, 1 << 40, None)
            assert st == binding.Q3A_EINVAL
    a = list(args)
    a[5] = 0
    assert lib.q3a_prefill_chunk(*a, 1, 4, 32, 8, 128, 64, 1e6, 1e-6, FAKE, 1 << 40,
                                 None) == binding.Q3A_EINVAL


def test_chunk_workspace_size(lib):
    assert binding.prefill_chunk_workspace_size(2, 100, 32, 8) >= 256 + 2 * 100 * 32 * 256
    assert binding.prefill_chunk_workspace_size(2, 100, 32, 8, 64) == 0


def test_device_pos_decode_host_checks(lib):
    """Argument errors the host can see are refused before any launch; the
    positions themselves are on the device and are not read here."""
    def call(**kw):
        a = dict(B=2, Hq=32, Hkv=8, d=128, S_max=64, theta=1e6, eps=1e-6, ws=FAKE,
                 ws_bytes=1 << 40, pos=FAKE)
        a.update(kw)
        return lib.q3a_decode_device_pos(FAKE, FAKE, FAKE, FAKE, FAKE, a["pos"], FAKE, FAKE, FAKE,
                                         a["B"], a["Hq"], a["Hkv"], a["d"], a["S_max"],
                                         a["theta"], a["eps"], a["ws"], a["ws_bytes"], None)
    assert call(d=64) == binding.Q3A_EINVAL
    assert call(Hq=12) == binding.Q3A_EINVAL
    assert call(pos=0) == binding.Q3A_EINVAL
    assert call(pos=FAKE + 2) == binding.Q3A_EINVAL
    assert call(ws_bytes=16) == binding.Q3A_EINVAL
    assert call(S_max=0) == binding.Q3A_EINVAL
    assert call(B=2049) == binding.Q3A_EINVAL
    assert call(B=0) == binding.Q3A_OK


def gated_call(lib, **kw):
    a = dict(B=1, T=4, Hq=16, Hkv=2, d=256, d_rot=64, theta=1e7, eps=1e-6, ws=FAKE,
             ws_bytes=1 << 40)
    a.update(kw)
    return lib.q3a_gated_prefill(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["B"], a["T"], a["Hq"],
                                 a["Hkv"], a["d"], a["d_rot"], a["theta"], a["eps"], a["ws"],
                                 a["ws_bytes"], None)


def test_gated_unsupported_group_is_notimpl(lib):
    # more than 16 query heads per KV head: a whole ratio, not implemented
    assert gated_call(lib, Hq=64, Hkv=2) == binding.Q3A_ENOTIMPL
    assert gated_call(lib, Hq=68, Hkv=2) == binding.Q3A_ENOTIMPL


@pytest.mark.parametrize("kw", [dict(d=128), dict(d_rot=8), dict(d_rot=-16), dict(d_rot=272),
                                dict(d_rot=65), dict(Hq=12, Hkv=5), dict(Hq=0, Hkv=1),
                                dict(Hq=190, Hkv=10), dict(eps=0.0), dict(theta=0.5),
                                dict(B=-1), dict(ws=FAKE + 16), dict(ws=0),
                                dict(ws_bytes=4096)])
def test_gated_prefill_rejects_bad_arguments(lib, kw):
    assert gated_call(lib, **kw) == binding.Q3A_EINVAL


def test_gated_prefill_empty_and_pointer_checks(lib):
    assert gated_call(lib, B=0) == binding.Q3A_OK
    assert gated_call(lib, T=0) == binding.Q3A_OK
    for i in range(6):
        for bad in (0, FAKE + 2):
            a = [FAKE] * 6
            a[i] = bad
            st = lib.q3a_gated_prefill(*a, 1, 4, 16, 2, 256, 64, 1e7, 1e-6, FAKE, 1 << 40, None)
            assert st == binding.Q3A_EINVAL
    # the two halves check the same way
    assert lib.q3a_gated_prefill_prologue(FAKE, FAKE, FAKE, FAKE, 1, 4, 16, 2, 256, 24, 1e7,
                                          1e-6, FAKE, 1 << 40, None) == binding.Q3A_EINVAL
    assert lib.q3a_gated_prefill_attention(FAKE, FAKE, FAKE + 8, 1, 4, 16, 2, 256, FAKE,
                                           1 << 40, None) == binding.Q3A_EINVAL


def test_gated_workspace_size(lib):
    B, T, Hq, Hkv = 4, 4096, 16, 2
    ws = binding.gated_prefill_workspace_size(B, T, Hq, Hkv)
    assert ws >= 256 + B * T * (Hq + Hkv) * 256 * 2
    assert binding.gated_prefill_workspace_size(B, T, Hq, Hkv, 128) == 0


def gated_decode_call(lib, start_pos, S_max=64, **kw):
    B = len(start_pos)
    sp = (ctypes.c_int32 * max(B, 1))(*start_pos)
    a = dict(Hq=16, Hkv=2, d=256, d_rot=64, theta=1e7, eps=1e-6, ws=FAKE, ws_bytes=1 << 40)
    a.update(kw)
    return lib.q3a_gated_decode(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.addressof(sp), FAKE, FAKE,
                                FAKE, B, a["Hq"], a["Hkv"], a["d"], a["d_rot"], S_max, a["theta"],
                                a["eps"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("sp", [[64], [-1], [3, 70]])
def test_gated_decode_context_overflow_is_erange(lib, sp):
    assert gated_decode_call(lib, sp) == binding.Q3A_ERANGE


def test_gated_decode_rejects_bad_arguments(lib):
    for kw in (dict(d=128), dict(d_rot=8), dict(d_rot=272), dict(eps=0.0), dict(theta=1.0),
               dict(ws=FAKE + 8), dict(ws_bytes=1024), dict(Hq=15, Hkv=2)):
        assert gated_decode_call(lib, [3], **kw) == binding.Q3A_EINVAL, kw
    assert gated_decode_call(lib, [3], Hq=34, Hkv=2) == binding.Q3A_ENOTIMPL
    assert gated_decode_call(lib, []) == binding.Q3A_OK
    ws = binding.gated_decode_workspace_size(64, 16, 2, 32768)
    assert ws >= 256 + 64 * 2 * 16 * 8 * (2 + 256) * 4  # 2048-key splits at d = 256


def test_gated_prefill_fill_host_checks(lib):
    def call(B=1, T=4, Hq=16, Hkv=2, d=256, d_rot=64, S_max=8, ws_bytes=1 << 40):
        return lib.q3a_gated_prefill_fill(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, T, Hq,
                                          Hkv, d, d_rot, S_max, 1e7, 1e-6, FAKE, ws_bytes, None)
    assert call(T=9, S_max=8) == binding.Q3A_ERANGE
    assert call(Hq=36, Hkv=2) == binding.Q3A_ENOTIMPL
    assert call(d=128) == binding.Q3A_EINVAL
    assert call(ws_bytes=1024) == binding.Q3A_EINVAL
    assert call(Hq=160, Hkv=20) == binding.Q3A_EINVAL  # 160 + 2*20 staged rows per token > 192
    assert call(T=0) == binding.Q3A_OK
    assert lib.q3a_gated_prefill_fill_workspace_size(2, 100, 16, 2, 256) >= 256 + 2 * 100 * 16 * 512


def test_gated_prefill_chunk_host_checks(lib):
    def call(sp=(3,), Tq=4, Hq=16, Hkv=2, d=256, d_rot=64, S_max=8, ws_bytes=1 << 40):
        B = len(sp)
        arr = (ctypes.c_int32 * max(B, 1))(*sp)
        return lib.q3a_gated_prefill_chunk(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.addressof(arr),
                                           FAKE, FAKE, FAKE, B, Tq, Hq, Hkv, d, d_rot, S_max,
                                           1e7, 1e-6, FAKE, ws_bytes, None)
    assert call(sp=(5,)) == binding.Q3A_ERANGE      # 5 + 4 > 8
    assert call(sp=(0, -1)) == binding.Q3A_ERANGE
    assert call(sp=(0, 5)) == binding.Q3A_ERANGE      # any sequence out of range
    assert call(Hq=36, Hkv=2) == binding.Q3A_ENOTIMPL
    for kw in (dict(d=128), dict(d_rot=8), dict(ws_bytes=1024), dict(Hq=15, Hkv=2),
               dict(Hq=160, Hkv=20), dict(S_max=0)):
        assert call(**kw) == binding.Q3A_EINVAL, kw
    assert call(sp=tuple([0] * 2049)) == binding.Q3A_EINVAL  # more sequences than one call takes
    assert call(Tq=0) == binding.Q3A_OK
    assert call(sp=()) == binding.Q3A_OK
    assert (lib.q3a_gated_prefill_chunk_workspace_size(2, 100, 16, 2, 256)
            == lib.q3a_gated_prefill_fill_workspace_size(2, 100, 16, 2, 256))


def test_selftest_validates_before_launching(lib):
    assert lib.q3a_selftest_bounded_wait(None, 256, 1000, 0, None) == binding.Q3A_EINVAL
    assert lib.q3a_selftest_bounded_wait(FAKE, 128, 1000, 0, None) == binding.Q3A_EINVAL
    assert lib.q3a_selftest_bounded_wait(FAKE + 4, 256, 1000, 0, None) == binding.Q3A_EINVAL
    assert lib.q3a_selftest_bounded_wait(FAKE, 256, 0, 0, None) == binding.Q3A_EINVAL
    assert lib.q3a_selftest_bounded_wait(FAKE, 256, 1 << 62, 0, None) == binding.Q3A_EINVAL
