"""Seeded synthetic inputs for the attention core (shared by tests and bench).

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and distributions of the workloads and names them. Both the
CUDA path and the CPU oracle are fed from here.

Recipe (all draws from a ``torch.Generator`` seeded with the workload's seed):
  prefill: Q [B,T,Hq,d], K [B,T,Hkv,d], V [B,T,Hkv,d] ~ N(0,1) drawn in fp32, in
           that order; then gamma_q, gamma_k ~ U(0.5, 1.5) [d]; then, when the
           workload asks for norm outliers, an independent Bernoulli(p) mask per
           (b,t,h) row for Q and then for K whose rows are multiplied by the
           scale in fp32. Everything is rounded to bf16 (round-to-nearest-even)
           at the end.
  decode:  start_pos [B] ~ U{lo, ..., hi-1} from a CPU generator; then cache K,
           cache V [B,Hkv,S_max,d] ~ N(0,1); then q [B,Hq,d], k_new, v_new
           [B,Hkv,d] ~ N(0,1); then gamma_q, gamma_k ~ U(0.5, 1.5). Cache rows
           start_pos[b] and later are set to NaN, so that a read of a row that
           the step may not read shows up in the output.
  chunk:   the prefill draws for whole prompts of sp_lo + T tokens (seeded as
           above); the first sp_lo tokens go into the caches through an earlier
           chunk, the last T are the timed chunk. Caches start as NaN.
  gated:   (Qwen3-Next / Qwen3.5 global attention) the query projection
           QG [B,T,Hq,2d] (per head: query, then gate), K [B,T,Hkv,d],
           V [B,T,Hkv,d] ~ N(0,1) in fp32, in that order; then the zero-centred
           norm weights w_q, w_k ~ U(-0.5, 0.5) [d] (scales 1 + w in [0.5, 1.5],
           the range of the gammas above); rounded to bf16 at the end.
  gated decode: start_pos as for decode; then cache K, cache V [B,Hkv,S_max,d]
           ~ N(0,1) (rows start_pos[b].. set to NaN); then QG [B,Hq,2d], k_new,
           v_new [B,Hkv,d] ~ N(0,1); then w_q, w_k ~ U(-0.5, 0.5).
  gated chunk: whole prompts of sp_lo + T tokens drawn as for gated; the first
           sp_lo go into the caches through an earlier chunk, the last T are
           the timed chunk. Caches start as NaN.

Large workloads are drawn on the GPU (``device="cuda"``) with torch's CUDA
generator; small ones on the CPU. Either way the draws are deterministic for a
given seed and device.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "prefill", "decode", "chunk", "gated", "gated_decode" or "gated_chunk"
    B: int
    Hq: int
    Hkv: int
    d: int = 128
    T: int = 0          # prefill (or chunk) tokens per sequence
    S_max: int = 0      # decode / chunk cache capacity
    sp_lo: int = 0      # decode start_pos range [sp_lo, sp_hi); chunk: its start position
    sp_hi: int = 0
    theta: float = 1e6
    eps: float = 1e-6
    seed: int = 0
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    d_r: int = 0        # gated: rotated leading coordinates per head
    note: str = field(default="", compare=False)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("qwen3-0.6b-prefill-b1-t128", "prefill", B=1, T=128, Hq=16, Hkv=8,
                 theta=1e6, seed=0,
                 note="Qwen3-0.6B-shaped tiny prefill, positions 0..127"),
        Workload("qwen3-8b-prefill-b4-t4096", "prefill", B=4, T=4096, Hq=32, Hkv=8,
                 theta=1e6, seed=1, outlier_frac=0.01, outlier_scale=30.0,
                 note="Qwen3-8B-shaped prefill, 1% of Q/K rows scaled x30"),
        Workload("qwen3-32b-prefill-b2-t8192", "prefill", B=2, T=8192, Hq=64, Hkv=8,
                 theta=1e6, seed=2, note="Qwen3-32B-shaped prefill"),
        Workload("qwen3-8b-decode-b64", "decode", B=64, Hq=32, Hkv=8, S_max=32768,
                 sp_lo=1024, sp_hi=32768, theta=1e6, seed=3,
                 note="Qwen3-8B-shaped decode, start_pos ~ U[1024, 32768)"),
        Workload("qwen3-8b-chunk-b4-t1024-at3072", "chunk", B=4, T=1024, Hq=32, Hkv=8,
                 S_max=4096, sp_lo=3072, sp_hi=3073, theta=1e6, seed=5,
                 note="Qwen3-8B-shaped chunked prefill: the last 1024 tokens of 4096-token "
                      "prompts whose first 3072 tokens are already in the cache"),
        Workload("qwen3-30b-a3b-prefill-b1-t32768", "prefill", B=1, T=32768, Hq=32, Hkv=4,
                 theta=1e7, seed=4, note="Qwen3-30B-A3B-shaped long-context prefill"),
        Workload("qwen3.5-0.8b-gated-b1-t300", "gated", B=1, T=300, Hq=8, Hkv=2, d=256,
                 d_r=64, theta=1e7, seed=6,
                 note="Qwen3.5-0.8B-shaped gated global attention, small (full parity)"),
        Workload("qwen3-next-80b-gated-b4-t4096", "gated", B=4, T=4096, Hq=16, Hkv=2, d=256,
                 d_r=64, theta=1e7, seed=7,
                 note="Qwen3-Next-80B-A3B-shaped gated global attention prefill"),
        Workload("qwen3.5-397b-gated-b1-t8192", "gated", B=1, T=8192, Hq=32, Hkv=2, d=256,
                 d_r=64, theta=1e7, seed=8,
                 note="Qwen3.5-397B-A17B-shaped gated global attention prefill (g = 16)"),
        Workload("qwen3-next-80b-gated-decode-b64", "gated_decode", B=64, Hq=16, Hkv=2, d=256,
                 S_max=32768, sp_lo=1024, sp_hi=32768, d_r=64, theta=1e7, seed=9,
                 note="Qwen3-Next-80B-A3B-shaped gated decode, start_pos ~ U[1024, 32768)"),
        Workload("qwen3-next-80b-gated-chunk-b4-t1024-at3072", "gated_chunk", B=4, T=1024,
                 Hq=16, Hkv=2, d=256, S_max=4096, sp_lo=3072, sp_hi=3073, d_r=64, theta=1e7,
                 seed=10,
                 note="Qwen3-Next-80B-A3B-shaped gated chunked prefill: the last 1024 tokens "
                      "of 4096-token prompts whose first 3072 tokens are already cached"),
    ]
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def prefill_inputs(B: int, T: int, Hq: int, Hkv: int, d: int = 128, seed: int = 0,
                   outlier_frac: float = 0.0, outlier_scale: float = 1.0,
                   device="cpu") -> dict:
    """Q, K, V, gamma_q, gamma_k as bf16 tensors on ``device``."""
    dev = torch.device(device)
    g = _gen(dev, seed)
    f32 = torch.float32
    q = torch.randn((B, T, Hq, d), generator=g, device=dev, dtype=f32)
    k = torch.randn((B, T, Hkv, d), generator=g, device=dev, dtype=f32)
    v = torch.randn((B, T, Hkv, d), generator=g, device=dev, dtype=f32)
    q_gamma = torch.rand((d,), generator=g, device=dev, dtype=f32) + 0.5
    k_gamma = torch.rand((d,), generator=g, device=dev, dtype=f32) + 0.5
    if outlier_frac > 0.0:
        mq = torch.rand((B, T, Hq), generator=g, device=dev, dtype=f32) < outlier_frac
        mk = torch.rand((B, T, Hkv), generator=g, device=dev, dtype=f32) < outlier_frac
        q[mq] *= outlier_scale
        k[mk] *= outlier_scale
    bf = torch.bfloat16
    return dict(q=q.to(bf), k=k.to(bf), v=v.to(bf), q_gamma=q_gamma.to(bf),
                k_gamma=k_gamma.to(bf))


def decode_inputs(B: int, Hq: int, Hkv: int, S_max: int, sp_lo: int, sp_hi: int,
                  d: int = 128, seed: int = 0, device="cpu", start_pos=None) -> dict:
    """Decode-step inputs. ``start_pos`` (host int32 [B]) is drawn unless given."""
    dev = torch.device(device)
    if start_pos is None:
        start_pos = torch.randint(sp_lo, sp_hi, (B,), generator=_gen("cpu", seed),
                                  dtype=torch.int64).to(torch.int32)
    else:
        start_pos = torch.as_tensor(start_pos, dtype=torch.int32).clone()
    g = _gen(dev, seed + 7919)
    bf = torch.bfloat16
    k_cache = torch.randn((B, Hkv, S_max, d), generator=g, device=dev, dtype=bf)
    v_cache = torch.randn((B, Hkv, S_max, d), generator=g, device=dev, dtype=bf)
    f32 = torch.float32
    q = torch.randn((B, Hq, d), generator=g, device=dev, dtype=f32)
    k_new = torch.randn((B, Hkv, d), generator=g, device=dev, dtype=f32)
    v_new = torch.randn((B, Hkv, d), generator=g, device=dev, dtype=f32)
    q_gamma = torch.rand((d,), generator=g, device=dev, dtype=f32) + 0.5
    k_gamma = torch.rand((d,), generator=g, device=dev, dtype=f32) + 0.5
    for b in range(B):
        p = int(start_pos[b])
        k_cache[b, :, p:, :] = float("nan")
        v_cache[b, :, p:, :] = float("nan")
    return dict(q=q.to(bf), k_new=k_new.to(bf), v_new=v_new.to(bf), k_cache=k_cache,
                v_cache=v_cache, start_pos=start_pos, q_gamma=q_gamma.to(bf),
                k_gamma=k_gamma.to(bf))


def gated_inputs(B: int, T: int, Hq: int, Hkv: int, d: int = 256, seed: int = 0,
                 device="cpu") -> dict:
    """QG (query|gate per head), K, V, w_q, w_k as bf16 tensors on ``device``."""
    dev = torch.device(device)
    g = _gen(dev, seed)
    f32 = torch.float32
    qg = torch.randn((B, T, Hq, 2 * d), generator=g, device=dev, dtype=f32)
    k = torch.randn((B, T, Hkv, d), generator=g, device=dev, dtype=f32)
    v = torch.randn((B, T, Hkv, d), generator=g, device=dev, dtype=f32)
    q_w = torch.rand((d,), generator=g, device=dev, dtype=f32) - 0.5
    k_w = torch.rand((d,), generator=g, device=dev, dtype=f32) - 0.5
    bf = torch.bfloat16
    return dict(qg=qg.to(bf), k=k.to(bf), v=v.to(bf), q_w=q_w.to(bf), k_w=k_w.to(bf))


def gated_decode_inputs(B: int, Hq: int, Hkv: int, S_max: int, sp_lo: int, sp_hi: int,
                        d: int = 256, seed: int = 0, device="cpu", start_pos=None) -> dict:
    """Gated decode-step inputs. ``start_pos`` (host int32 [B]) is drawn unless given."""
    dev = torch.device(device)
    if start_pos is None:
        start_pos = torch.randint(sp_lo, sp_hi, (B,), generator=_gen("cpu", seed),
                                  dtype=torch.int64).to(torch.int32)
    else:
        start_pos = torch.as_tensor(start_pos, dtype=torch.int32).clone()
    g = _gen(dev, seed + 7919)
    bf = torch.bfloat16
    k_cache = torch.randn((B, Hkv, S_max, d), generator=g, device=dev, dtype=bf)
    v_cache = torch.randn((B, Hkv, S_max, d), generator=g, device=dev, dtype=bf)
    f32 = torch.float32
    qg = torch.randn((B, Hq, 2 * d), generator=g, device=dev, dtype=f32)
    k_new = torch.randn((B, Hkv, d), generator=g, device=dev, dtype=f32)
    v_new = torch.randn((B, Hkv, d), generator=g, device=dev, dtype=f32)
    q_w = torch.rand((d,), generator=g, device=dev, dtype=f32) - 0.5
    k_w = torch.rand((d,), generator=g, device=dev, dtype=f32) - 0.5
    for b in range(B):
        p = int(start_pos[b])
        k_cache[b, :, p:, :] = float("nan")
        v_cache[b, :, p:, :] = float("nan")
    return dict(qg=qg.to(bf), k_new=k_new.to(bf), v_new=v_new.to(bf), k_cache=k_cache,
                v_cache=v_cache, start_pos=start_pos, q_w=q_w.to(bf), k_w=k_w.to(bf))


def workload_inputs(w: Workload, device="cpu") -> dict:
    if w.kind == "gated_decode":
        return gated_decode_inputs(w.B, w.Hq, w.Hkv, w.S_max, w.sp_lo, w.sp_hi, w.d, w.seed,
                                   device=device)
    if w.kind == "gated":
        return gated_inputs(w.B, w.T, w.Hq, w.Hkv, w.d, w.seed, device=device)
    if w.kind == "gated_chunk":  # whole prompts; the caller splits them
        return gated_inputs(w.B, w.sp_lo + w.T, w.Hq, w.Hkv, w.d, w.seed, device=device)
    if w.kind == "chunk":  # whole prompts; the caller splits them
        return prefill_inputs(w.B, w.sp_lo + w.T, w.Hq, w.Hkv, w.d, w.seed, device=device)
    if w.kind == "prefill":
        return prefill_inputs(w.B, w.T, w.Hq, w.Hkv, w.d, w.seed, w.outlier_frac,
                              w.outlier_scale, device=device)
    return decode_inputs(w.B, w.Hq, w.Hkv, w.S_max, w.sp_lo, w.sp_hi, w.d, w.seed,
                         device=device)
