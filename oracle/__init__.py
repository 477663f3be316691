"""CPU oracle of the Qwen3 attention core (QK-Norm -> RoPE -> causal GQA),
and of the gated global-attention layer of Qwen3-Next / Qwen3.5.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product library never
imports, links or runs anything here, and this package imports nothing from it.

The arithmetic lives in ``q3a_oracle.c`` (plain fp64 loops, see its header for
the definition and the page passages each step follows). This module compiles
it with gcc and wraps it with ctypes. Inputs are bf16 torch CPU tensors (their
exact values are widened to fp64); outputs are fp64 torch tensors.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, invariants and a separately written brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q3a_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libq3a_oracle.so")
_lock = threading.Lock()
_lib = None

_u16p = ctypes.c_void_p
_f64p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libq3a_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
            lib.q3a_oracle_set_threads.argtypes = [i]
            lib.q3a_oracle_threads.restype = i
            lib.q3a_oracle_rmsnorm_row.argtypes = [_u16p, _u16p, i, d, _f64p]
            lib.q3a_oracle_rope_row.argtypes = [_f64p, i, d, d]
            lib.q3a_oracle_qknorm_rope.argtypes = [_u16p, _u16p, i, i, i, i, l, d, d, _f64p]
            lib.q3a_oracle_qknorm_rope.restype = i
            lib.q3a_oracle_prefill.argtypes = [_u16p] * 5 + [i] * 5 + [d, d, _f64p]
            lib.q3a_oracle_prefill.restype = i
            lib.q3a_oracle_prefill_rounded.argtypes = [_u16p] * 5 + [i] * 5 + [d, d, i, _f64p]
            lib.q3a_oracle_prefill_rounded.restype = i
            lib.q3a_oracle_round_bf16.argtypes = [_f64p, l, _f64p]
            lib.q3a_oracle_prefill_rows.argtypes = ([_u16p] * 5 + [i] * 5 + [d, d, l]
                                                    + [ctypes.c_void_p] * 3 + [_f64p])
            lib.q3a_oracle_prefill_rows.restype = i
            lib.q3a_oracle_decode.argtypes = ([_u16p] * 5 + [ctypes.c_void_p] + [_u16p] * 2
                                              + [i] * 4 + [l, d, d, ctypes.c_void_p,
                                                            _f64p, _f64p])
            lib.q3a_oracle_decode.restype = i
            lib.q3a_oracle_prefill_chunk.argtypes = ([_u16p] * 5 + [ctypes.c_void_p] + [_u16p] * 2
                                                     + [i] * 5 + [l, d, d, _f64p, _f64p])
            lib.q3a_oracle_prefill_chunk.restype = i
            lib.q3a_oracle_zc_rmsnorm_row.argtypes = [_u16p, _u16p, i, d, _f64p]
            lib.q3a_oracle_partial_rope_row.argtypes = [_f64p, i, i, d, d]
            lib.q3a_oracle_partial_rope_row.restype = i
            lib.q3a_oracle_gated_prefill.argtypes = [_u16p] * 5 + [i] * 6 + [d, d, _f64p]
            lib.q3a_oracle_gated_prefill.restype = i
            lib.q3a_oracle_gated_prefill_rows.argtypes = ([_u16p] * 5 + [i] * 6 + [d, d, l]
                                                          + [ctypes.c_void_p] * 3 + [_f64p])
            lib.q3a_oracle_gated_prefill_rows.restype = i
            lib.q3a_oracle_gated_qknorm_rope.argtypes = [_u16p, l, _u16p, i, i, i, i, i, l, d,
                                                         d, _f64p]
            lib.q3a_oracle_gated_qknorm_rope.restype = i
            lib.q3a_oracle_gated_decode.argtypes = ([_u16p] * 5 + [ctypes.c_void_p] + [_u16p] * 2
                                                    + [i] * 5 + [l, d, d, _f64p, _f64p])
            lib.q3a_oracle_gated_decode.restype = i
            lib.q3a_oracle_gated_prefill_chunk.argtypes = ([_u16p] * 5 + [ctypes.c_void_p]
                                                           + [_u16p] * 2 + [i] * 6
                                                           + [l, d, d, _f64p, _f64p])
            lib.q3a_oracle_gated_prefill_chunk.restype = i
            _lib = lib
    return _lib


def _bf16(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.bfloat16 or t.device.type != "cpu":
        raise TypeError(f"{name}: expected a bf16 CPU tensor, got {t.dtype} on {t.device}")
    return t.contiguous()


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def set_threads(n: int) -> None:
    """Number of OpenMP threads the oracle uses (0 = OpenMP default)."""
    _load().q3a_oracle_set_threads(int(n))


def threads() -> int:
    """Threads the oracle's parallel loops run with."""
    return int(_load().q3a_oracle_threads())


def rmsnorm_row(x: torch.Tensor, gamma: torch.Tensor, eps: float) -> torch.Tensor:
    """Step 1 on one row: x / sqrt(mean(x^2) + eps) * gamma, fp64."""
    x, gamma = _bf16(x, "x"), _bf16(gamma, "gamma")
    d = x.numel()
    y = torch.empty(d, dtype=torch.float64)
    _load().q3a_oracle_rmsnorm_row(_ptr(x), _ptr(gamma), d, float(eps), _ptr(y))
    return y


def rope_row(y: torch.Tensor, pos: float, theta: float) -> torch.Tensor:
    """Step 2 on one fp64 row (returns a rotated copy)."""
    out = y.to(torch.float64).contiguous().clone()
    _load().q3a_oracle_rope_row(_ptr(out), out.numel(), float(pos), float(theta))
    return out


def qknorm_rope(x: torch.Tensor, gamma: torch.Tensor, theta: float, eps: float,
                pos0: int = 0) -> torch.Tensor:
    """Steps 1-2 on x [B, T, H, d]; row (b, t, h) is rotated at pos0 + t. fp64 out."""
    x, gamma = _bf16(x, "x"), _bf16(gamma, "gamma")
    B, T, H, d = x.shape
    out = torch.empty((B, T, H, d), dtype=torch.float64)
    rc = _load().q3a_oracle_qknorm_rope(_ptr(x), _ptr(gamma), B, T, H, d, int(pos0),
                                        float(theta), float(eps), _ptr(out))
    if rc:
        raise ValueError(f"oracle qknorm_rope rejected its arguments ({rc})")
    return out


def prefill(q, k, v, q_gamma, k_gamma, theta: float, eps: float) -> torch.Tensor:
    """Full causal prefill; q [B,T,Hq,d], k/v [B,T,Hkv,d] -> fp64 [B,T,Hq,d]."""
    q, k, v = _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v")
    q_gamma, k_gamma = _bf16(q_gamma, "q_gamma"), _bf16(k_gamma, "k_gamma")
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    out = torch.empty((B, T, Hq, d), dtype=torch.float64)
    rc = _load().q3a_oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(q_gamma), _ptr(k_gamma),
                                    B, T, Hq, Hkv, d, float(theta), float(eps), _ptr(out))
    if rc:
        raise ValueError(f"oracle prefill failed ({rc})")
    return out


def prefill_rounded(q, k, v, q_gamma, k_gamma, theta: float, eps: float,
                    roundings: int = 1) -> torch.Tensor:
    """The full causal prefill with qhat and khat rounded to bf16 (nearest,
    ties to even): after RoPE only (``roundings=1``, the bf16 operands of the
    attention products), or after the norm and again after RoPE
    (``roundings=2``, the casts of §7.2.1's RMSNorm and apply_rope). Every other
    step in fp64. -> fp64 [B,T,Hq,d]."""
    q, k, v = _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v")
    q_gamma, k_gamma = _bf16(q_gamma, "q_gamma"), _bf16(k_gamma, "k_gamma")
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    out = torch.empty((B, T, Hq, d), dtype=torch.float64)
    rc = _load().q3a_oracle_prefill_rounded(_ptr(q), _ptr(k), _ptr(v), _ptr(q_gamma),
                                            _ptr(k_gamma), B, T, Hq, Hkv, d, float(theta),
                                            float(eps), int(roundings), _ptr(out))
    if rc:
        raise ValueError(f"oracle prefill_rounded failed ({rc})")
    return out


def round_bf16(x: torch.Tensor) -> torch.Tensor:
    """fp64 values rounded to the nearest bf16 value (ties to even), as fp64."""
    x = x.to(torch.float64).contiguous()
    y = torch.empty_like(x)
    _load().q3a_oracle_round_bf16(_ptr(x), x.numel(), _ptr(y))
    return y


def prefill_rows(q, k, v, q_gamma, k_gamma, theta: float, eps: float,
                 rows: torch.Tensor) -> torch.Tensor:
    """Sampled causal prefill. rows: int32 [n, 3] of (b, t, h). -> fp64 [n, d]."""
    q, k, v = _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v")
    q_gamma, k_gamma = _bf16(q_gamma, "q_gamma"), _bf16(k_gamma, "k_gamma")
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    rows = rows.to(torch.int32)
    rb, rt, rh = (rows[:, c].contiguous() for c in range(3))
    n = rows.shape[0]
    out = torch.empty((n, d), dtype=torch.float64)
    rc = _load().q3a_oracle_prefill_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(q_gamma),
                                         _ptr(k_gamma), B, T, Hq, Hkv, d, float(theta),
                                         float(eps), n, _ptr(rb), _ptr(rt), _ptr(rh),
                                         _ptr(out))
    if rc:
        raise ValueError(f"oracle prefill_rows failed ({rc})")
    return out


def decode(q, k_new, v_new, k_cache, v_cache, start_pos, q_gamma, k_gamma,
           theta: float, eps: float, select=None):
    """One decode step. Returns (out fp64 [B,Hq,d], appended key row fp64 [B,Hkv,d]).

    ``select``: optional bool [B]; only those sequences are computed (others
    are left as zeros).
    """
    q, k_new, v_new = _bf16(q, "q"), _bf16(k_new, "k_new"), _bf16(v_new, "v_new")
    k_cache, v_cache = _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    q_gamma, k_gamma = _bf16(q_gamma, "q_gamma"), _bf16(k_gamma, "k_gamma")
    B, Hq, d = q.shape
    Hkv, S_max = k_cache.shape[1], k_cache.shape[2]
    sp = torch.as_tensor(start_pos, dtype=torch.int32).contiguous()
    sel = None if select is None else torch.as_tensor(select, dtype=torch.uint8).contiguous()
    out = torch.zeros((B, Hq, d), dtype=torch.float64)
    k_row = torch.zeros((B, Hkv, d), dtype=torch.float64)
    rc = _load().q3a_oracle_decode(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                   _ptr(v_cache), _ptr(sp), _ptr(q_gamma), _ptr(k_gamma),
                                   B, Hq, Hkv, d, S_max, float(theta), float(eps),
                                   None if sel is None else _ptr(sel), _ptr(out), _ptr(k_row))
    if rc:
        raise ValueError(f"oracle decode failed ({rc})")
    return out, k_row


def prefill_chunk(q, k, v, k_cache, v_cache, start_pos, q_gamma, k_gamma, theta: float,
                  eps: float):
    """Chunked prefill. q [B,Tq,Hq,d], k/v [B,Tq,Hkv,d]; caches [B,Hkv,S_max,d].

    Returns (out fp64 [B,Tq,Hq,d], appended key rows fp64 [B,Tq,Hkv,d]).
    """
    q, k, v = _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v")
    k_cache, v_cache = _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    q_gamma, k_gamma = _bf16(q_gamma, "q_gamma"), _bf16(k_gamma, "k_gamma")
    B, Tq, Hq, d = q.shape
    Hkv, S_max = k_cache.shape[1], k_cache.shape[2]
    sp = torch.as_tensor(start_pos, dtype=torch.int32).contiguous()
    out = torch.zeros((B, Tq, Hq, d), dtype=torch.float64)
    k_rows = torch.zeros((B, Tq, Hkv, d), dtype=torch.float64)
    rc = _load().q3a_oracle_prefill_chunk(_ptr(q), _ptr(k), _ptr(v), _ptr(k_cache),
                                          _ptr(v_cache), _ptr(sp), _ptr(q_gamma), _ptr(k_gamma),
                                          B, Tq, Hq, Hkv, d, S_max, float(theta), float(eps),
                                          _ptr(out), _ptr(k_rows))
    if rc:
        raise ValueError(f"oracle prefill_chunk failed ({rc})")
    return out, k_rows


# ---------------------------------------------------------------------------
# The gated global-attention layer of Qwen3-Next / Qwen3.5 (steps g1-g5 of
# q3a_oracle.c): per-head query/gate split, zero-centred norm (1 + w), partial
# rotary on the first d_r coordinates, causal GQA attention, sigmoid gate.
# ---------------------------------------------------------------------------

def zc_rmsnorm_row(x: torch.Tensor, w: torch.Tensor, eps: float) -> torch.Tensor:
    """g2 on one row: x / sqrt(mean(x^2) + eps) * (1 + w), fp64."""
    x, w = _bf16(x, "x"), _bf16(w, "w")
    d = x.numel()
    y = torch.empty(d, dtype=torch.float64)
    _load().q3a_oracle_zc_rmsnorm_row(_ptr(x), _ptr(w), d, float(eps), _ptr(y))
    return y


def partial_rope_row(y: torch.Tensor, d_r: int, pos: float, theta: float) -> torch.Tensor:
    """g3 on one fp64 row: rotate-half RoPE of the first d_r coordinates only."""
    out = y.to(torch.float64).contiguous().clone()
    rc = _load().q3a_oracle_partial_rope_row(_ptr(out), out.numel(), int(d_r), float(pos),
                                             float(theta))
    if rc:
        raise ValueError(f"oracle partial_rope_row rejected d_r={d_r}")
    return out


def gated_prefill(qg, k, v, q_w, k_w, d_r: int, theta: float, eps: float) -> torch.Tensor:
    """Gated causal prefill. qg [B,T,Hq,2d] (per head: query, then gate),
    k/v [B,T,Hkv,d], q_w/k_w [d] zero-centred weights -> fp64 [B,T,Hq,d]."""
    qg, k, v = _bf16(qg, "qg"), _bf16(k, "k"), _bf16(v, "v")
    q_w, k_w = _bf16(q_w, "q_w"), _bf16(k_w, "k_w")
    B, T, Hq, d2 = qg.shape
    Hkv, d = k.shape[2], k.shape[3]
    if d2 != 2 * d:
        raise ValueError(f"qg last dim {d2} != 2 * {d}")
    out = torch.empty((B, T, Hq, d), dtype=torch.float64)
    rc = _load().q3a_oracle_gated_prefill(_ptr(qg), _ptr(k), _ptr(v), _ptr(q_w), _ptr(k_w),
                                          B, T, Hq, Hkv, d, int(d_r), float(theta), float(eps),
                                          _ptr(out))
    if rc:
        raise ValueError(f"oracle gated_prefill failed ({rc})")
    return out


def gated_prefill_rows(qg, k, v, q_w, k_w, d_r: int, theta: float, eps: float,
                       rows: torch.Tensor) -> torch.Tensor:
    """Sampled gated prefill. rows: int32 [n, 3] of (b, t, h) -> fp64 [n, d]."""
    qg, k, v = _bf16(qg, "qg"), _bf16(k, "k"), _bf16(v, "v")
    q_w, k_w = _bf16(q_w, "q_w"), _bf16(k_w, "k_w")
    B, T, Hq, d2 = qg.shape
    Hkv, d = k.shape[2], k.shape[3]
    if d2 != 2 * d:
        raise ValueError(f"qg last dim {d2} != 2 * {d}")
    rows = rows.to(torch.int32)
    rb, rt, rh = (rows[:, c].contiguous() for c in range(3))
    n = rows.shape[0]
    out = torch.empty((n, d), dtype=torch.float64)
    rc = _load().q3a_oracle_gated_prefill_rows(_ptr(qg), _ptr(k), _ptr(v), _ptr(q_w),
                                               _ptr(k_w), B, T, Hq, Hkv, d, int(d_r),
                                               float(theta), float(eps), n, _ptr(rb),
                                               _ptr(rt), _ptr(rh), _ptr(out))
    if rc:
        raise ValueError(f"oracle gated_prefill_rows failed ({rc})")
    return out


def gated_qknorm_rope(x, w, d: int, d_r: int, theta: float, eps: float,
                      pos0: int = 0) -> torch.Tensor:
    """g2 then g3 on the first d elements of every row of x [B, T, H, S] (S = 2d
    for the query halves of the query/gate projection, d for keys); row
    (b, t, h) at position pos0 + t. -> fp64 [B, T, H, d]."""
    x, w = _bf16(x, "x"), _bf16(w, "w")
    B, T, H, S = x.shape
    out = torch.empty((B, T, H, d), dtype=torch.float64)
    rc = _load().q3a_oracle_gated_qknorm_rope(_ptr(x), S, _ptr(w), B, T, H, d, int(d_r),
                                              int(pos0), float(theta), float(eps), _ptr(out))
    if rc:
        raise ValueError(f"oracle gated_qknorm_rope rejected its arguments ({rc})")
    return out


def gated_decode(qg, k_new, v_new, k_cache, v_cache, start_pos, q_w, k_w, d_r: int,
                 theta: float, eps: float):
    """One gated decode step. qg [B,Hq,2d] (per head: query, then gate), k_new/v_new
    [B,Hkv,d], caches [B,Hkv,S_max,d]. Returns (out fp64 [B,Hq,d], appended key
    row fp64 [B,Hkv,d])."""
    qg, k_new, v_new = _bf16(qg, "qg"), _bf16(k_new, "k_new"), _bf16(v_new, "v_new")
    k_cache, v_cache = _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    q_w, k_w = _bf16(q_w, "q_w"), _bf16(k_w, "k_w")
    B, Hq, d2 = qg.shape
    Hkv, S_max, d = k_cache.shape[1], k_cache.shape[2], k_cache.shape[3]
    if d2 != 2 * d:
        raise ValueError(f"qg last dim {d2} != 2 * {d}")
    sp = torch.as_tensor(start_pos, dtype=torch.int32).contiguous()
    out = torch.zeros((B, Hq, d), dtype=torch.float64)
    k_row = torch.zeros((B, Hkv, d), dtype=torch.float64)
    rc = _load().q3a_oracle_gated_decode(_ptr(qg), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                         _ptr(v_cache), _ptr(sp), _ptr(q_w), _ptr(k_w), B, Hq,
                                         Hkv, d, int(d_r), S_max, float(theta), float(eps),
                                         _ptr(out), _ptr(k_row))
    if rc:
        raise ValueError(f"oracle gated_decode failed ({rc})")
    return out, k_row


def gated_prefill_chunk(qg, k, v, k_cache, v_cache, start_pos, q_w, k_w, d_r: int,
                        theta: float, eps: float):
    """Gated chunk of Tq tokens per sequence against the caches. qg [B,Tq,Hq,2d],
    k/v [B,Tq,Hkv,d], caches [B,Hkv,S_max,d]. Returns (out fp64 [B,Tq,Hq,d],
    the chunk's keys fp64 [B,Tq,Hkv,d])."""
    qg, k, v = _bf16(qg, "qg"), _bf16(k, "k"), _bf16(v, "v")
    k_cache, v_cache = _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache")
    q_w, k_w = _bf16(q_w, "q_w"), _bf16(k_w, "k_w")
    B, Tq, Hq, d2 = qg.shape
    Hkv, S_max, d = k_cache.shape[1], k_cache.shape[2], k_cache.shape[3]
    if d2 != 2 * d:
        raise ValueError(f"qg last dim {d2} != 2 * {d}")
    sp = torch.as_tensor(start_pos, dtype=torch.int32).contiguous()
    out = torch.zeros((B, Tq, Hq, d), dtype=torch.float64)
    k_rows = torch.zeros((B, Tq, Hkv, d), dtype=torch.float64)
    rc = _load().q3a_oracle_gated_prefill_chunk(_ptr(qg), _ptr(k), _ptr(v), _ptr(k_cache),
                                                _ptr(v_cache), _ptr(sp), _ptr(q_w), _ptr(k_w),
                                                B, Tq, Hq, Hkv, d, int(d_r), S_max,
                                                float(theta), float(eps), _ptr(out),
                                                _ptr(k_rows))
    if rc:
        raise ValueError(f"oracle gated_prefill_chunk failed ({rc})")
    return out, k_rows
