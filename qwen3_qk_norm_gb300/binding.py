"""ctypes binding of libq3a (include/q3a.h): argument marshalling only.

Every step of the attention core runs in the CUDA library; this module checks
tensor dtypes, shapes and devices, passes raw device pointers and the current
torch stream, and turns a non-zero status into ``Q3AError``. It has no
fallback: if ``libq3a.so`` is missing, ``load()`` raises ``ImportError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

Q3A_OK, Q3A_EINVAL, Q3A_ERANGE, Q3A_ECUDA, Q3A_ETIMEOUT, Q3A_ENOTIMPL = range(6)
STATUS_NAMES = {0: "Q3A_OK", 1: "Q3A_EINVAL", 2: "Q3A_ERANGE", 3: "Q3A_ECUDA",
                4: "Q3A_ETIMEOUT", 5: "Q3A_ENOTIMPL"}
EXPORTED = ["q3a_status_string", "q3a_qknorm_rope", "q3a_prefill_workspace_size", "q3a_prefill",
            "q3a_prefill_prologue", "q3a_prefill_attention", "q3a_prefill_chunk_workspace_size",
            "q3a_prefill_chunk", "q3a_decode_workspace_size",
            "q3a_decode", "q3a_decode_device_pos", "q3a_decode_noalloc",
            "q3a_last_device_error", "q3a_gated_prefill_workspace_size", "q3a_gated_prefill",
            "q3a_gated_prefill_prologue", "q3a_gated_prefill_attention",
            "q3a_gated_decode_workspace_size", "q3a_gated_decode",
            "q3a_gated_decode_device_pos", "q3a_gated_prefill_fill_workspace_size",
            "q3a_gated_prefill_fill", "q3a_gated_prefill_chunk_workspace_size",
            "q3a_gated_prefill_chunk", "q3a_selftest_bounded_wait"]

_lock = threading.Lock()
_lib = None


class Q3AError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} "
                         f"({_load_quiet_status_string(status)})")


def _load_quiet_status_string(status: int) -> str:
    try:
        return load().q3a_status_string(status).decode()
    except Exception:  # noqa: BLE001 - message only
        return "?"


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libq3a.so (build it first with ``qwen3_qk_norm_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"libq3a.so not found at {p}: run qwen3_qk_norm_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i, d, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_float, ctypes.c_size_t
        lib.q3a_status_string.argtypes = [i]
        lib.q3a_status_string.restype = ctypes.c_char_p
        lib.q3a_qknorm_rope.argtypes = [vp, vp, vp, i, i, i, i, i, d, f, vp]
        lib.q3a_qknorm_rope.restype = i
        lib.q3a_prefill_workspace_size.argtypes = [i, i, i, i, i]
        lib.q3a_prefill_workspace_size.restype = sz
        lib.q3a_prefill.argtypes = [vp] * 6 + [i] * 5 + [d, f, vp, sz, vp]
        lib.q3a_prefill.restype = i
        lib.q3a_prefill_prologue.argtypes = [vp] * 3 + [i] * 5 + [d, f, vp, sz, vp]
        lib.q3a_prefill_prologue.restype = i
        lib.q3a_prefill_attention.argtypes = [vp] * 4 + [i] * 5 + [f, vp, sz, vp]
        lib.q3a_prefill_attention.restype = i
        lib.q3a_prefill_chunk_workspace_size.argtypes = [i] * 5
        lib.q3a_prefill_chunk_workspace_size.restype = sz
        lib.q3a_prefill_chunk.argtypes = [vp] * 9 + [i] * 6 + [d, f, vp, sz, vp]
        lib.q3a_prefill_chunk.restype = i
        lib.q3a_decode_workspace_size.argtypes = [i] * 5
        lib.q3a_decode_workspace_size.restype = sz
        lib.q3a_decode.argtypes = [vp] * 9 + [i] * 5 + [d, f, vp, sz, vp]
        lib.q3a_decode.restype = i
        lib.q3a_decode_device_pos.argtypes = [vp] * 9 + [i] * 5 + [d, f, vp, sz, vp]
        lib.q3a_decode_device_pos.restype = i
        lib.q3a_decode_noalloc.argtypes = [vp] * 9 + [i] * 5 + [d, f, vp]
        lib.q3a_decode_noalloc.restype = i
        lib.q3a_last_device_error.argtypes = [vp, vp]
        lib.q3a_last_device_error.restype = i
        lib.q3a_selftest_bounded_wait.argtypes = [vp, sz, ctypes.c_longlong, i, vp]
        lib.q3a_selftest_bounded_wait.restype = i
        lib.q3a_gated_prefill_workspace_size.argtypes = [i] * 5
        lib.q3a_gated_prefill_workspace_size.restype = sz
        lib.q3a_gated_prefill.argtypes = [vp] * 6 + [i] * 6 + [d, f, vp, sz, vp]
        lib.q3a_gated_prefill.restype = i
        lib.q3a_gated_prefill_prologue.argtypes = [vp] * 4 + [i] * 6 + [d, f, vp, sz, vp]
        lib.q3a_gated_prefill_prologue.restype = i
        lib.q3a_gated_prefill_attention.argtypes = [vp] * 3 + [i] * 5 + [vp, sz, vp]
        lib.q3a_gated_prefill_attention.restype = i
        lib.q3a_gated_decode_workspace_size.argtypes = [i] * 5
        lib.q3a_gated_decode_workspace_size.restype = sz
        lib.q3a_gated_decode.argtypes = [vp] * 9 + [i] * 6 + [d, f, vp, sz, vp]
        lib.q3a_gated_decode.restype = i
        lib.q3a_gated_decode_device_pos.argtypes = [vp] * 9 + [i] * 6 + [d, f, vp, sz, vp]
        lib.q3a_gated_decode_device_pos.restype = i
        lib.q3a_gated_prefill_fill_workspace_size.argtypes = [i] * 5
        lib.q3a_gated_prefill_fill_workspace_size.restype = sz
        lib.q3a_gated_prefill_fill.argtypes = [vp] * 8 + [i] * 7 + [d, f, vp, sz, vp]
        lib.q3a_gated_prefill_fill.restype = i
        lib.q3a_gated_prefill_chunk_workspace_size.argtypes = [i] * 5
        lib.q3a_gated_prefill_chunk_workspace_size.restype = sz
        lib.q3a_gated_prefill_chunk.argtypes = [vp] * 9 + [i] * 7 + [d, f, vp, sz, vp]
        lib.q3a_gated_prefill_chunk.restype = i
        _lib = lib
        return lib


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(t: torch.Tensor, name: str, shape=None, dtype=torch.bfloat16) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: expected a CUDA tensor, got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _raise(status: int, what: str) -> None:
    if status != Q3A_OK:
        raise Q3AError(status, what)


def qknorm_rope(x: torch.Tensor, gamma: torch.Tensor, theta: float, eps: float,
                pos0: int = 0, out: torch.Tensor | None = None) -> torch.Tensor:
    """RoPE_{pos0+t}(RMSNorm(x) * gamma) for x [B, T, H, 128] bf16."""
    B, T, H, d = x.shape
    _check(x, "x")
    _check(gamma, "gamma", (d,))
    if out is None:
        out = torch.empty_like(x)
    _check(out, "out", x.shape)
    st = load().q3a_qknorm_rope(x.data_ptr(), gamma.data_ptr(), out.data_ptr(), B, T, H, d,
                                int(pos0), float(theta), float(eps), _stream(x.device))
    _raise(st, "q3a_qknorm_rope")
    return out


def prefill_workspace_size(B: int, T: int, Hq: int, Hkv: int, d: int = 128) -> int:
    return int(load().q3a_prefill_workspace_size(B, T, Hq, Hkv, d))


def prefill(q, k, v, q_gamma, k_gamma, theta: float, eps: float, out=None,
            workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Causal prefill: q [B,T,Hq,128], k/v [B,T,Hkv,128] bf16 -> out [B,T,Hq,128] bf16."""
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    _check(q, "q")
    _check(k, "k", (B, T, Hkv, d))
    _check(v, "v", (B, T, Hkv, d))
    _check(q_gamma, "q_gamma", (d,))
    _check(k_gamma, "k_gamma", (d,))
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", q.shape)
    need = prefill_workspace_size(B, T, Hq, Hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(), q_gamma.data_ptr(),
                            k_gamma.data_ptr(), out.data_ptr(), B, T, Hq, Hkv, d, float(theta),
                            float(eps), workspace.data_ptr(), workspace.numel(),
                            _stream(q.device))
    _raise(st, "q3a_prefill")
    return out


def prefill_prologue(k, q_gamma, k_gamma, Hq: int, theta: float, eps: float,
                     workspace: torch.Tensor) -> None:
    """Steps 1-2 of prefill for the keys into ``workspace`` (see q3a_prefill_prologue)."""
    B, T, Hkv, d = k.shape
    _check(k, "k")
    _check(q_gamma, "q_gamma", (d,))
    _check(k_gamma, "k_gamma", (d,))
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_prefill_prologue(k.data_ptr(), q_gamma.data_ptr(), k_gamma.data_ptr(), B, T,
                                     Hq, Hkv, d, float(theta), float(eps), workspace.data_ptr(),
                                     workspace.numel(), _stream(k.device))
    _raise(st, "q3a_prefill_prologue")


def prefill_attention(q, v, q_gamma, out, eps: float, workspace: torch.Tensor) -> torch.Tensor:
    """The query norm and attention of prefill, with the keys from ``workspace``
    (see q3a_prefill_attention)."""
    B, T, Hq, d = q.shape
    Hkv = v.shape[2]
    _check(q, "q")
    _check(v, "v", (B, T, Hkv, d))
    _check(q_gamma, "q_gamma", (d,))
    _check(out, "out", (B, T, Hq, d))
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_prefill_attention(q.data_ptr(), v.data_ptr(), q_gamma.data_ptr(),
                                      out.data_ptr(), B, T, Hq, Hkv, d, float(eps),
                                      workspace.data_ptr(), workspace.numel(), _stream(q.device))
    _raise(st, "q3a_prefill_attention")
    return out


def prefill_chunk_workspace_size(B: int, Tq: int, Hq: int, Hkv: int, d: int = 128) -> int:
    return int(load().q3a_prefill_chunk_workspace_size(B, Tq, Hq, Hkv, d))


def _host_positions(start_pos, B: int) -> torch.Tensor:
    sp = torch.as_tensor(start_pos, dtype=torch.int32).contiguous()
    if sp.device.type != "cpu" or sp.numel() != B:
        raise ValueError("start_pos: expected a host array of B int32")
    return sp


def prefill_chunk(q, k, v, k_cache, v_cache, start_pos, q_gamma, k_gamma, theta: float,
                  eps: float, out=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Prefill of a chunk of Tq tokens per sequence against the caches, which
    it extends by the chunk's normalised, rotated keys and its values.

    q [B,Tq,Hq,128], k/v [B,Tq,Hkv,128] bf16; caches [B,Hkv,S_max,128] bf16;
    start_pos: host int32 [B], position of each sequence's first chunk token.
    """
    B, Tq, Hq, d = q.shape
    Hkv, S_max = k_cache.shape[1], k_cache.shape[2]
    _check(q, "q")
    _check(k, "k", (B, Tq, Hkv, d))
    _check(v, "v", (B, Tq, Hkv, d))
    _check(k_cache, "k_cache", (B, Hkv, S_max, d))
    _check(v_cache, "v_cache", (B, Hkv, S_max, d))
    _check(q_gamma, "q_gamma", (d,))
    _check(k_gamma, "k_gamma", (d,))
    sp = _host_positions(start_pos, B)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", q.shape)
    need = prefill_chunk_workspace_size(B, Tq, Hq, Hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_prefill_chunk(q.data_ptr(), k.data_ptr(), v.data_ptr(), k_cache.data_ptr(),
                                  v_cache.data_ptr(), sp.data_ptr(), q_gamma.data_ptr(),
                                  k_gamma.data_ptr(), out.data_ptr(), B, Tq, Hq, Hkv, d, S_max,
                                  float(theta), float(eps), workspace.data_ptr(),
                                  workspace.numel(), _stream(q.device))
    _raise(st, "q3a_prefill_chunk")
    return out


def decode_workspace_size(B: int, Hq: int, Hkv: int, S_max: int, d: int = 128) -> int:
    return int(load().q3a_decode_workspace_size(B, Hq, Hkv, d, S_max))


def decode(q, k_new, v_new, k_cache, v_cache, start_pos, q_gamma, k_gamma, theta: float,
           eps: float, out=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """One decode step; appends the new key/value at start_pos[b] in the caches.

    q [B,Hq,128], k_new/v_new [B,Hkv,128] bf16; caches [B,Hkv,S_max,128] bf16;
    start_pos: host int32 [B] (list, numpy or CPU tensor).
    """
    B, Hq, d = q.shape
    Hkv, S_max = k_cache.shape[1], k_cache.shape[2]
    _check(q, "q")
    _check(k_new, "k_new", (B, Hkv, d))
    _check(v_new, "v_new", (B, Hkv, d))
    _check(k_cache, "k_cache", (B, Hkv, S_max, d))
    _check(v_cache, "v_cache", (B, Hkv, S_max, d))
    _check(q_gamma, "q_gamma", (d,))
    _check(k_gamma, "k_gamma", (d,))
    sp = _host_positions(start_pos, B)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", q.shape)
    need = decode_workspace_size(B, Hq, Hkv, S_max, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_decode(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                           v_cache.data_ptr(), sp.data_ptr(), q_gamma.data_ptr(),
                           k_gamma.data_ptr(), out.data_ptr(), B, Hq, Hkv, d, S_max,
                           float(theta), float(eps), workspace.data_ptr(), workspace.numel(),
                           _stream(q.device))
    _raise(st, "q3a_decode")
    return out


def decode_device_pos(q, k_new, v_new, k_cache, v_cache, start_pos, q_gamma, k_gamma,
                      theta: float, eps: float, out=None,
                      workspace: torch.Tensor | None = None) -> torch.Tensor:
    """One decode step with the positions in device memory (start_pos: CUDA
    int32 [B]); capturable into a CUDA graph. An out-of-range position makes
    the step write nothing and last_device_error() return Q3A_ERANGE."""
    B, Hq, d = q.shape
    Hkv, S_max = k_cache.shape[1], k_cache.shape[2]
    _check(q, "q")
    _check(k_new, "k_new", (B, Hkv, d))
    _check(v_new, "v_new", (B, Hkv, d))
    _check(k_cache, "k_cache", (B, Hkv, S_max, d))
    _check(v_cache, "v_cache", (B, Hkv, S_max, d))
    _check(q_gamma, "q_gamma", (d,))
    _check(k_gamma, "k_gamma", (d,))
    _check(start_pos, "start_pos", (B,), dtype=torch.int32)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", q.shape)
    need = decode_workspace_size(B, Hq, Hkv, S_max, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_decode_device_pos(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                      k_cache.data_ptr(), v_cache.data_ptr(),
                                      start_pos.data_ptr(), q_gamma.data_ptr(),
                                      k_gamma.data_ptr(), out.data_ptr(), B, Hq, Hkv, d, S_max,
                                      float(theta), float(eps), workspace.data_ptr(),
                                      workspace.numel(), _stream(q.device))
    _raise(st, "q3a_decode_device_pos")
    return out


def last_device_error(workspace: torch.Tensor | None) -> int:
    """Status from the error word a call left in its workspace (synchronises).
    ``None`` reads the error word of q3a_decode_noalloc on the current device."""
    if workspace is None:
        dev = torch.device("cuda", torch.cuda.current_device())
        return int(load().q3a_last_device_error(None, _stream(dev)))
    return int(load().q3a_last_device_error(workspace.data_ptr(), _stream(workspace.device)))


def selftest_bounded_wait(workspace: torch.Tensor, limit_cycles: int, arrive: bool) -> None:
    """Launches the bounded-wait self-test (one block waiting on an mbarrier
    that completes only if ``arrive``); read the outcome with
    ``last_device_error(workspace)``."""
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_selftest_bounded_wait(workspace.data_ptr(), workspace.numel(),
                                          int(limit_cycles), int(bool(arrive)),
                                          _stream(workspace.device))
    _raise(st, "q3a_selftest_bounded_wait")


# ---------------------------------------------------------------------------
# gated global attention of Qwen3-Next / Qwen3.5 (include/q3a.h q3a_gated_*)
# ---------------------------------------------------------------------------

def gated_prefill_workspace_size(B: int, T: int, Hq: int, Hkv: int, d: int = 256) -> int:
    return int(load().q3a_gated_prefill_workspace_size(B, T, Hq, Hkv, d))


def _gated_shapes(qg, k):
    B, T, Hq, d2 = qg.shape
    d = d2 // 2
    Hkv = k.shape[2]
    return B, T, Hq, Hkv, d


def gated_prefill(qg, k, v, q_w, k_w, d_rot: int, theta: float, eps: float, out=None,
                  workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Gated causal prefill: qg [B,T,Hq,512] (per head: query, then gate),
    k/v [B,T,Hkv,256], q_w/k_w [256] zero-centred weights -> out [B,T,Hq,256]."""
    B, T, Hq, Hkv, d = _gated_shapes(qg, k)
    _check(qg, "qg")
    _check(k, "k", (B, T, Hkv, d))
    _check(v, "v", (B, T, Hkv, d))
    _check(q_w, "q_w", (d,))
    _check(k_w, "k_w", (d,))
    if out is None:
        out = torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device=qg.device)
    _check(out, "out", (B, T, Hq, d))
    need = gated_prefill_workspace_size(B, T, Hq, Hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=qg.device)
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_gated_prefill(qg.data_ptr(), k.data_ptr(), v.data_ptr(), q_w.data_ptr(),
                                  k_w.data_ptr(), out.data_ptr(), B, T, Hq, Hkv, d, int(d_rot),
                                  float(theta), float(eps), workspace.data_ptr(),
                                  workspace.numel(), _stream(qg.device))
    _raise(st, "q3a_gated_prefill")
    return out


def gated_prefill_prologue(qg, k, q_w, k_w, d_rot: int, theta: float, eps: float,
                           workspace: torch.Tensor) -> None:
    """The norm + partial-RoPE kernel of gated_prefill into ``workspace``."""
    B, T, Hq, Hkv, d = _gated_shapes(qg, k)
    _check(qg, "qg")
    _check(k, "k", (B, T, Hkv, d))
    _check(q_w, "q_w", (d,))
    _check(k_w, "k_w", (d,))
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_gated_prefill_prologue(qg.data_ptr(), k.data_ptr(), q_w.data_ptr(),
                                           k_w.data_ptr(), B, T, Hq, Hkv, d, int(d_rot),
                                           float(theta), float(eps), workspace.data_ptr(),
                                           workspace.numel(), _stream(qg.device))
    _raise(st, "q3a_gated_prefill_prologue")


def gated_prefill_attention(qg, v, out, workspace: torch.Tensor) -> torch.Tensor:
    """The gated attention kernel of gated_prefill, from ``workspace``."""
    B, T, Hq, d2 = qg.shape
    Hkv, d = v.shape[2], v.shape[3]
    _check(qg, "qg")
    _check(v, "v", (B, T, Hkv, d))
    _check(out, "out", (B, T, Hq, d))
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_gated_prefill_attention(qg.data_ptr(), v.data_ptr(), out.data_ptr(), B, T,
                                            Hq, Hkv, d, workspace.data_ptr(), workspace.numel(),
                                            _stream(v.device))
    _raise(st, "q3a_gated_prefill_attention")
    return out


def gated_decode_workspace_size(B: int, Hq: int, Hkv: int, S_max: int, d: int = 256) -> int:
    return int(load().q3a_gated_decode_workspace_size(B, Hq, Hkv, d, S_max))


def gated_decode(qg, k_new, v_new, k_cache, v_cache, start_pos, q_w, k_w, d_rot: int,
                 theta: float, eps: float, out=None,
                 workspace: torch.Tensor | None = None) -> torch.Tensor:
    """One gated decode step: qg [B,Hq,512] (query | gate per head), k_new/v_new
    [B,Hkv,256], caches [B,Hkv,S_max,256] (row start_pos[b] is appended), start_pos
    host int32 [B] -> out [B,Hq,256]."""
    B, Hq, d2 = qg.shape
    d = d2 // 2
    Hkv, S_max = k_cache.shape[1], k_cache.shape[2]
    _check(qg, "qg")
    _check(k_new, "k_new", (B, Hkv, d))
    _check(v_new, "v_new", (B, Hkv, d))
    _check(k_cache, "k_cache", (B, Hkv, S_max, d))
    _check(v_cache, "v_cache", (B, Hkv, S_max, d))
    _check(q_w, "q_w", (d,))
    _check(k_w, "k_w", (d,))
    sp = _host_positions(start_pos, B)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=qg.device)
    _check(out, "out", (B, Hq, d))
    need = gated_decode_workspace_size(B, Hq, Hkv, S_max, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=qg.device)
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_gated_decode(qg.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                 k_cache.data_ptr(), v_cache.data_ptr(), sp.data_ptr(),
                                 q_w.data_ptr(), k_w.data_ptr(), out.data_ptr(), B, Hq, Hkv, d,
                                 int(d_rot), S_max, float(theta), float(eps),
                                 workspace.data_ptr(), workspace.numel(), _stream(qg.device))
    _raise(st, "q3a_gated_decode")
    return out


def gated_decode_device_pos(qg, k_new, v_new, k_cache, v_cache, start_pos, q_w, k_w,
                            d_rot: int, theta: float, eps: float, out=None,
                            workspace: torch.Tensor | None = None) -> torch.Tensor:
    """gated_decode with start_pos a CUDA int32 [B] tensor (capturable in a CUDA
    graph); an out-of-range position writes nothing and is reported by
    last_device_error(workspace) as Q3A_ERANGE."""
    B, Hq, d2 = qg.shape
    d = d2 // 2
    Hkv, S_max = k_cache.shape[1], k_cache.shape[2]
    _check(qg, "qg")
    _check(k_new, "k_new", (B, Hkv, d))
    _check(v_new, "v_new", (B, Hkv, d))
    _check(k_cache, "k_cache", (B, Hkv, S_max, d))
    _check(v_cache, "v_cache", (B, Hkv, S_max, d))
    _check(q_w, "q_w", (d,))
    _check(k_w, "k_w", (d,))
    _check(start_pos, "start_pos", (B,), dtype=torch.int32)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device=qg.device)
    _check(out, "out", (B, Hq, d))
    need = gated_decode_workspace_size(B, Hq, Hkv, S_max, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=qg.device)
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_gated_decode_device_pos(qg.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                            k_cache.data_ptr(), v_cache.data_ptr(),
                                            start_pos.data_ptr(), q_w.data_ptr(), k_w.data_ptr(),
                                            out.data_ptr(), B, Hq, Hkv, d, int(d_rot), S_max,
                                            float(theta), float(eps), workspace.data_ptr(),
                                            workspace.numel(), _stream(qg.device))
    _raise(st, "q3a_gated_decode_device_pos")
    return out


def gated_prefill_fill(qg, k, v, k_cache, v_cache, q_w, k_w, d_rot: int, theta: float,
                       eps: float, out=None, workspace: torch.Tensor | None = None
                       ) -> torch.Tensor:
    """gated_prefill of a prompt that also writes the normalised, rotated keys and
    the values into rows 0..T-1 of the caches [B,Hkv,S_max,256]."""
    B, T, Hq, Hkv, d = _gated_shapes(qg, k)
    S_max = k_cache.shape[2]
    _check(qg, "qg")
    _check(k, "k", (B, T, Hkv, d))
    _check(v, "v", (B, T, Hkv, d))
    _check(k_cache, "k_cache", (B, Hkv, S_max, d))
    _check(v_cache, "v_cache", (B, Hkv, S_max, d))
    _check(q_w, "q_w", (d,))
    _check(k_w, "k_w", (d,))
    if out is None:
        out = torch.empty((B, T, Hq, d), dtype=torch.bfloat16, device=qg.device)
    _check(out, "out", (B, T, Hq, d))
    need = int(load().q3a_gated_prefill_fill_workspace_size(B, T, Hq, Hkv, d))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=qg.device)
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_gated_prefill_fill(qg.data_ptr(), k.data_ptr(), v.data_ptr(),
                                       k_cache.data_ptr(), v_cache.data_ptr(), q_w.data_ptr(),
                                       k_w.data_ptr(), out.data_ptr(), B, T, Hq, Hkv, d,
                                       int(d_rot), S_max, float(theta), float(eps),
                                       workspace.data_ptr(), workspace.numel(),
                                       _stream(qg.device))
    _raise(st, "q3a_gated_prefill_fill")
    return out


def gated_prefill_chunk_workspace_size(B: int, Tq: int, Hq: int, Hkv: int, d: int = 256) -> int:
    return int(load().q3a_gated_prefill_chunk_workspace_size(B, Tq, Hq, Hkv, d))


def gated_prefill_chunk(qg, k, v, k_cache, v_cache, start_pos, q_w, k_w, d_rot: int,
                        theta: float, eps: float, out=None,
                        workspace: torch.Tensor | None = None) -> torch.Tensor:
    """A chunk of Tq tokens per sequence of the gated layer against its caches,
    which it extends by the chunk's normalised, rotated keys and its values.

    qg [B,Tq,Hq,512], k/v [B,Tq,Hkv,256] bf16; caches [B,Hkv,S_max,256] bf16;
    start_pos: host int32 [B], position of each sequence's first chunk token.
    """
    B, Tq, Hq, Hkv, d = _gated_shapes(qg, k)
    S_max = k_cache.shape[2]
    _check(qg, "qg")
    _check(k, "k", (B, Tq, Hkv, d))
    _check(v, "v", (B, Tq, Hkv, d))
    _check(k_cache, "k_cache", (B, Hkv, S_max, d))
    _check(v_cache, "v_cache", (B, Hkv, S_max, d))
    _check(q_w, "q_w", (d,))
    _check(k_w, "k_w", (d,))
    sp = _host_positions(start_pos, B)
    if out is None:
        out = torch.empty((B, Tq, Hq, d), dtype=torch.bfloat16, device=qg.device)
    _check(out, "out", (B, Tq, Hq, d))
    need = gated_prefill_chunk_workspace_size(B, Tq, Hq, Hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=qg.device)
    _check(workspace, "workspace", dtype=torch.uint8)
    st = load().q3a_gated_prefill_chunk(qg.data_ptr(), k.data_ptr(), v.data_ptr(),
                                        k_cache.data_ptr(), v_cache.data_ptr(), sp.data_ptr(),
                                        q_w.data_ptr(), k_w.data_ptr(), out.data_ptr(), B, Tq, Hq,
                                        Hkv, d, int(d_rot), S_max, float(theta), float(eps),
                                        workspace.data_ptr(), workspace.numel(),
                                        _stream(qg.device))
    _raise(st, "q3a_gated_prefill_chunk")
    return out
