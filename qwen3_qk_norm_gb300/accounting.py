"""Work accounting of the attention core: algorithmic flops and bytes.

These are the denominators of the benchmark's roofline figures, counted from
the definition of each step, not from what a kernel happens to move.
"""
from __future__ import annotations


def prefill_flops(B: int, T: int, Hq: int, d: int = 128) -> int:
    """Algorithmic flops of causal prefill: QK^T and PV at 2d each per unmasked pair."""
    return 4 * d * Hq * B * T * (T + 1) // 2


def chunk_flops(start_pos, Tq: int, Hq: int, d: int = 128) -> int:
    """Algorithmic flops of a chunk of Tq tokens per sequence after start_pos[b]
    cached tokens: token t sees start_pos[b] + t + 1 keys, 4d flops per pair."""
    pairs = sum(Tq * int(p) + Tq * (Tq + 1) // 2 for p in start_pos)
    return 4 * d * Hq * pairs


def decode_bytes(start_pos, Hq: int, Hkv: int, d: int = 128) -> int:
    """Algorithmic HBM bytes of one decode step.

    Reads: cached K and V rows 0..start_pos[b]-1 of every (b, kv); q, k_new,
    v_new; the two gammas. Writes: the appended K and V rows and the output.
    """
    sp = [int(x) for x in start_pos]
    B = len(sp)
    row = d * 2
    cache_read = sum(sp) * Hkv * 2 * row
    new_in = B * (Hq + 2 * Hkv) * row + 2 * row
    writes = B * 2 * Hkv * row + B * Hq * row
    return cache_read + new_in + writes


def gated_decode_bytes(start_pos, Hq: int, Hkv: int, d: int = 256) -> int:
    """Algorithmic HBM bytes of one gated decode step: as decode_bytes, with
    the query/gate rows (2d per head) read instead of d-wide queries."""
    sp = [int(x) for x in start_pos]
    B = len(sp)
    row = d * 2
    cache_read = sum(sp) * Hkv * 2 * row
    new_in = B * (2 * Hq + 2 * Hkv) * row + 2 * row
    writes = B * 2 * Hkv * row + B * Hq * row
    return cache_read + new_in + writes


def kv_cache_bytes_per_token(n_layers: int, Hkv: int, d: int = 128, elem_bytes: int = 2) -> int:
    """K and V bytes one token occupies in a cache of ``n_layers`` layers."""
    return n_layers * Hkv * d * 2 * elem_bytes
