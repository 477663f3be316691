"""Whole-output parity at full size: every workload the benchmark runs, launched
as the benchmark launches it, compared element by element over its ENTIRE
output with the fp64 oracle run in full (no sampled rows).

Bar: bf16 outputs within max-abs 2e-2 and mean-abs 2e-3 of the oracle; the
rows a decode appends within one bf16 ulp of the oracle's normalised, rotated
key, and the appended values bit-exact.

The oracle runs on all host cores (several minutes for the 32768-token
prefill); each test prints its max-abs / mean-abs and the oracle's wall time.
"""
import time

import pytest
import torch

import oracle
from qwen3_qk_norm_gb300 import binding, inputs
from qwen3_qk_norm_gb300.inputs import WORKLOADS
from gpu_util import assert_close_attention, assert_within_one_ulp

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _report(name, mx, mean, oracle_s):
    print(f"\nFULL-PARITY {name}: max-abs {mx:.3e} mean-abs {mean:.3e} "
          f"(oracle {oracle_s:.1f} s on {oracle.threads()} threads)", flush=True)


@pytest.mark.parametrize("name", ["qwen3-0.6b-prefill-b1-t128", "qwen3-8b-prefill-b4-t4096",
                                  "qwen3-32b-prefill-b2-t8192",
                                  "qwen3-30b-a3b-prefill-b1-t32768"])
def test_prefill_workload_whole_output(cuda_lib, name):
    w = WORKLOADS[name]
    x = inputs.workload_inputs(w, device="cuda")
    out = binding.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], w.theta, w.eps)
    torch.cuda.synchronize()
    got = out.cpu()
    del out
    cpu = {k: t.cpu() for k, t in x.items()}
    del x
    t0 = time.perf_counter()
    ref = oracle.prefill(cpu["q"], cpu["k"], cpu["v"], cpu["q_gamma"], cpu["k_gamma"], w.theta,
                         w.eps)
    dt = time.perf_counter() - t0
    mx, mean = assert_close_attention(got, ref, name)
    _report(name, mx, mean, dt)


def test_decode_workload_all_sequences(cuda_lib):
    """Batch 64, start_pos ~ U[1024, 32768): all 64 sequences' outputs, and
    every appended K and V row."""
    w = WORKLOADS["qwen3-8b-decode-b64"]
    x = inputs.workload_inputs(w, device="cuda")
    cpu = {k: (t.cpu() if k != "start_pos" else t) for k, t in x.items()}  # before the append
    out = binding.decode(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                         x["start_pos"], x["q_gamma"], x["k_gamma"], w.theta, w.eps)
    torch.cuda.synchronize()
    got = out.cpu()
    sp = x["start_pos"].tolist()
    b_idx = torch.arange(w.B)
    p_idx = torch.tensor(sp)
    k_app = x["k_cache"][b_idx, :, p_idx].cpu()  # [B, Hkv, d]
    v_app = x["v_cache"][b_idx, :, p_idx].cpu()
    del x
    t0 = time.perf_counter()
    ref, k_row = oracle.decode(cpu["q"], cpu["k_new"], cpu["v_new"], cpu["k_cache"],
                               cpu["v_cache"], cpu["start_pos"], cpu["q_gamma"], cpu["k_gamma"],
                               w.theta, w.eps)
    dt = time.perf_counter() - t0
    mx, mean = assert_close_attention(got, ref, w.name)
    assert_within_one_ulp(k_app, k_row, "appended keys")
    assert torch.equal(v_app, cpu["v_new"])
    _report(w.name, mx, mean, dt)


def test_chunk_workload_whole_chunk(cuda_lib):
    """The chunked-prefill workload: each prompt's first 3072 tokens written
    into the caches by a chunk from position 0, then the last 1024 tokens as
    the measured chunk; its whole output against rows 3072..4095 of the
    oracle's prefill of the entire prompt."""
    w = WORKLOADS["qwen3-8b-chunk-b4-t1024-at3072"]
    x = inputs.workload_inputs(w, device="cuda")
    p0 = w.sp_lo
    kc = torch.full((w.B, w.Hkv, w.S_max, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    sl = lambda t, a, b: t[:, a:b].contiguous()  # noqa: E731
    binding.prefill_chunk(sl(x["q"], 0, p0), sl(x["k"], 0, p0), sl(x["v"], 0, p0), kc, vc,
                          [0] * w.B, x["q_gamma"], x["k_gamma"], w.theta, w.eps)
    out = binding.prefill_chunk(sl(x["q"], p0, None), sl(x["k"], p0, None),
                                sl(x["v"], p0, None), kc, vc, [p0] * w.B, x["q_gamma"],
                                x["k_gamma"], w.theta, w.eps)
    torch.cuda.synchronize()
    got = out.cpu()
    cpu = {k: t.cpu() for k, t in x.items()}
    del x, kc, vc, out
    t0 = time.perf_counter()
    ref = oracle.prefill(cpu["q"], cpu["k"], cpu["v"], cpu["q_gamma"], cpu["k_gamma"], w.theta,
                         w.eps)[:, p0:]
    dt = time.perf_counter() - t0
    mx, mean = assert_close_attention(got, ref, w.name)
    _report(w.name, mx, mean, dt)


@pytest.mark.parametrize("name", ["qwen3.5-0.8b-gated-b1-t300", "qwen3-next-80b-gated-b4-t4096",
                                  "qwen3.5-397b-gated-b1-t8192"])
def test_gated_workload_whole_output(cuda_lib, name):
    w = WORKLOADS[name]
    x = inputs.workload_inputs(w, device="cuda")
    out = binding.gated_prefill(x["qg"], x["k"], x["v"], x["q_w"], x["k_w"], w.d_r, w.theta,
                                w.eps)
    torch.cuda.synchronize()
    got = out.cpu()
    cpu = {k: t.cpu() for k, t in x.items()}
    del x, out
    t0 = time.perf_counter()
    ref = oracle.gated_prefill(cpu["qg"], cpu["k"], cpu["v"], cpu["q_w"], cpu["k_w"], w.d_r,
                               w.theta, w.eps)
    dt = time.perf_counter() - t0
    mx, mean = assert_close_attention(got, ref, name)
    _report(name, mx, mean, dt)


def test_gated_decode_workload_all_sequences(cuda_lib):
    w = WORKLOADS["qwen3-next-80b-gated-decode-b64"]
    x = inputs.workload_inputs(w, device="cuda")
    cpu = {k: (t.cpu() if k != "start_pos" else t) for k, t in x.items()}
    out = binding.gated_decode(x["qg"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                               x["start_pos"], x["q_w"], x["k_w"], w.d_r, w.theta, w.eps)
    torch.cuda.synchronize()
    got = out.cpu()
    b_idx = torch.arange(w.B)
    p_idx = torch.tensor(x["start_pos"].tolist())
    k_app = x["k_cache"][b_idx, :, p_idx].cpu()
    v_app = x["v_cache"][b_idx, :, p_idx].cpu()
    del x
    t0 = time.perf_counter()
    ref, k_row = oracle.gated_decode(cpu["qg"], cpu["k_new"], cpu["v_new"], cpu["k_cache"],
                                     cpu["v_cache"], cpu["start_pos"], cpu["q_w"], cpu["k_w"],
                                     w.d_r, w.theta, w.eps)
    dt = time.perf_counter() - t0
    mx, mean = assert_close_attention(got, ref, w.name)
    assert_within_one_ulp(k_app, k_row, "appended keys")
    assert torch.equal(v_app, cpu["v_new"])
    _report(w.name, mx, mean, dt)


def test_gated_chunk_workload_whole_chunk(cuda_lib):
    """As the chunk workload, on the gated layer: the last 1024 tokens of
    4096-token prompts against rows 3072..4095 of the oracle's gated prefill of
    the entire prompt."""
    w = WORKLOADS["qwen3-next-80b-gated-chunk-b4-t1024-at3072"]
    x = inputs.workload_inputs(w, device="cuda")
    p0 = w.sp_lo
    kc = torch.full((w.B, w.Hkv, w.S_max, w.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    sl = lambda t, a, b: t[:, a:b].contiguous()  # noqa: E731
    binding.gated_prefill_chunk(sl(x["qg"], 0, p0), sl(x["k"], 0, p0), sl(x["v"], 0, p0), kc, vc,
                                [0] * w.B, x["q_w"], x["k_w"], w.d_r, w.theta, w.eps)
    out = binding.gated_prefill_chunk(sl(x["qg"], p0, None), sl(x["k"], p0, None),
                                      sl(x["v"], p0, None), kc, vc, [p0] * w.B, x["q_w"],
                                      x["k_w"], w.d_r, w.theta, w.eps)
    torch.cuda.synchronize()
    got = out.cpu()
    cpu = {k: t.cpu() for k, t in x.items()}
    del x, kc, vc, out
    t0 = time.perf_counter()
    ref = oracle.gated_prefill(cpu["qg"], cpu["k"], cpu["v"], cpu["q_w"], cpu["k_w"], w.d_r,
                               w.theta, w.eps)[:, p0:]
    dt = time.perf_counter() - t0
    mx, mean = assert_close_attention(got, ref, w.name)
    _report(w.name, mx, mean, dt)
