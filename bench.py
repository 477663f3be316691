"""Benchmark of the Qwen3 attention core on GB300: causal prefill TFLOP/s and
decode GB/s, each against the measured roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on rank 0. A step is one q3a_prefill (QK-Norm + RoPE prologue,
then causal GQA attention) over the Qwen3-8B-shaped prefill workload (B=4,
T=4096, Hq=32, Hkv=8), inputs resident in HBM; ``value`` is its algorithmic
TFLOP/s (unmasked causal pairs only). The same run times the Qwen3-8B-shaped
decode workload (batch 64, start_pos in [1024, 32768)) in GB/s under "decode".
With N > 1 (torchrun) every rank runs its own copy of the workload (weak
scaling, no data-path collective); the time is the max over ranks.

``--impl reference`` times the fp64 CPU oracle on bounded samples of the same
workload (the only reference this method has: the pages give no code to run).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from qwen3_qk_norm_gb300 import accounting, inputs  # noqa: E402
from qwen3_qk_norm_gb300.inputs import WORKLOADS  # noqa: E402

METRIC = "causal prefill attention TFLOP/s and decode GB/s at 1 GB300, % of roofline"
PREFILL_WORKLOAD = "qwen3-8b-prefill-b4-t4096"
DECODE_WORKLOAD = "qwen3-8b-decode-b64"
CHUNK_WORKLOAD = "qwen3-8b-chunk-b4-t1024-at3072"
GATED_WORKLOAD = "qwen3-next-80b-gated-b4-t4096"
GATED_DECODE_WORKLOAD = "qwen3-next-80b-gated-decode-b64"
GATED_CHUNK_WORKLOAD = "qwen3-next-80b-gated-chunk-b4-t1024-at3072"
# the prefill workloads reported beside the headline one
EXTRA_PREFILL_WORKLOADS = ["qwen3-0.6b-prefill-b1-t128", "qwen3-32b-prefill-b2-t8192",
                           "qwen3-30b-a3b-prefill-b1-t32768"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 2 ** 20


# ----------------------------------------------------------------------------
# distributed plumbing (host logic; covered by the gloo tests)
# ----------------------------------------------------------------------------
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int, device=None):
    if world > 1:
        if device is not None and device.type == "cuda":
            torch.distributed.barrier(device_ids=[device.index])
        else:
            torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's value (times are reported as the max over ranks)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Weak scaling: every rank processes the same units; the job's rate is the
    sum of the units over the slowest rank's time."""
    return units_per_rank * world / seconds_max


# ----------------------------------------------------------------------------
# measurement helpers
# ----------------------------------------------------------------------------
def measured_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: torch.device, period_ms: int = 50):
        self.proc = None
        self.lines: list[str] = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:  # noqa: BLE001
            sel = ["-i", str(device.index or 0)]
        self.cmd = ["nvidia-smi"] + sel + ["--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                           f"-lms={period_ms}"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [s for s in sm if s > 0.5 * max(sm)]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


CSRC = os.path.join(ROOT, "qwen3_qk_norm_gb300", "csrc")
KERNEL_SOURCES = {  # the kernel's file and every header it includes
    "prefill_attention_kernel": ["prefill_attention.cu", "q3a_device.cuh", "q3a_internal.h"],
    "qknorm_rope_kernel": ["qknorm_rope.cu", "q3a_rope.cuh", "q3a_device.cuh", "q3a_internal.h"],
    "decode_split_kernel": ["decode_attention.cu", "q3a_rope.cuh", "q3a_device.cuh",
                            "q3a_internal.h"],
    "gated_attention_pair_kernel": ["gated_attention_pair.cu", "q3a_pair.cuh", "q3a_device.cuh",
                                    "q3a_internal.h"],
    "gated_prologue_kernel": ["gated_prologue.cu", "q3a_rope.cuh", "q3a_device.cuh",
                              "q3a_internal.h"],
    "decode_split_kernel<256>": ["decode_attention.cu", "q3a_rope.cuh", "q3a_device.cuh",
                                 "q3a_internal.h"],
    "gated_attention_pair_kernel<chunk>": ["gated_attention_pair.cu", "q3a_pair.cuh",
                                           "q3a_device.cuh", "q3a_internal.h"],
    "prefill_attention_kernel<chunk>": ["prefill_attention.cu", "q3a_device.cuh",
                                        "q3a_internal.h"],
}


def source_sha(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    sources are unchanged since that capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("source_sha") != source_sha(kernel):
        return None
    return float(rec["dram_bytes_per_launch"])


def synchronize_all(device):
    torch.cuda.synchronize(device)


# ----------------------------------------------------------------------------
# our implementation
# ----------------------------------------------------------------------------
def bench_prefill(binding, device, steps: int, warmup: int, world: int,
                  name: str = PREFILL_WORKLOAD):
    w = WORKLOADS[name]
    x = inputs.workload_inputs(w, device=device)
    out = torch.empty_like(x["q"])
    ws = torch.empty(binding.prefill_workspace_size(w.B, w.T, w.Hq, w.Hkv), dtype=torch.uint8,
                     device=device)
    stream = torch.cuda.current_stream(device)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        binding.prefill_prologue(x["k"], x["q_gamma"], x["k_gamma"], w.Hq, w.theta, w.eps, ws)
        if ev is not None:
            ev[1].record(stream)
        binding.prefill_attention(x["q"], x["v"], x["q_gamma"], out, w.eps, ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(warmup):
        step()
    # the step: back-to-back steps with events only around them (the kernels
    # of consecutive launches may overlap their start and end)
    barrier(world, device)
    synchronize_all(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step()
    t1.record(stream)
    synchronize_all(device)
    barrier(world, device)
    total_ms = t0.elapsed_time(t1)
    # each kernel alone: events between the two launches of every step
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    synchronize_all(device)
    for i in range(steps):
        step(evs[i])
    synchronize_all(device)
    k1_ms = [e[0].elapsed_time(e[1]) for e in evs]
    k2_ms = [e[1].elapsed_time(e[2]) for e in evs]
    status = binding.last_device_error(ws)
    if status != 0:
        raise RuntimeError(f"prefill device error word: {status}")
    return w, x, total_ms / steps, statistics.mean(k1_ms), statistics.mean(k2_ms)


def bench_prefill_e2e(binding, device, w, steps: int):
    """The step through q3a_prefill with host buffers: every step copies its
    inputs from pinned host memory to the device and its output back, inside
    the timed region. Three streams and two buffer sets pipeline the steps:
    step i+1's inputs travel while step i computes and step i-1's output
    returns; a buffer is refilled only after the step that used it is done."""
    xc = inputs.workload_inputs(w, device=device)
    n_buf = 2
    host = [{k: t.to("cpu").pin_memory() for k, t in xc.items()} for _ in range(n_buf)]
    dev = [{k: torch.empty_like(t) for k, t in xc.items()} for _ in range(n_buf)]
    outs = [torch.empty_like(xc["q"]) for _ in range(n_buf)]
    out_host = [torch.empty(xc["q"].shape, dtype=xc["q"].dtype, pin_memory=True)
                for _ in range(n_buf)]
    del xc
    ws = torch.empty(binding.prefill_workspace_size(w.B, w.T, w.Hq, w.Hkv), dtype=torch.uint8,
                     device=device)
    h2d = sum(t.numel() * t.element_size() for t in host[0].values())
    d2h = outs[0].numel() * outs[0].element_size()
    s_in, s_comp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev = {n: [torch.cuda.Event() for _ in range(n_buf)] for n in ("in", "comp", "out")}
    used = [False] * n_buf

    def step(i):
        j = i % n_buf
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(ev["comp"][j])  # step i-2 has read these inputs
            for k in dev[j]:
                dev[j][k].copy_(host[j][k], non_blocking=True)
            ev["in"][j].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev["in"][j])
            if used[j]:
                s_comp.wait_event(ev["out"][j])  # step i-2's output has left
            d = dev[j]
            binding.prefill(d["q"], d["k"], d["v"], d["q_gamma"], d["k_gamma"], w.theta, w.eps,
                            out=outs[j], workspace=ws)
            ev["comp"][j].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][j])
            out_host[j].copy_(outs[j], non_blocking=True)
            ev["out"][j].record(s_out)
        used[j] = True

    for i in range(n_buf + 1):  # warm-up: both buffer sets, three steps
        step(i)
    synchronize_all(device)
    # three timed passes of `steps` pipelined steps; the median pass is
    # reported, so one slow stretch of the shared host link does not decide it
    passes = []
    for _ in range(3):
        t0 = time.perf_counter()
        for i in range(steps):
            step(i)
        synchronize_all(device)
        passes.append((time.perf_counter() - t0) / steps)
    dt = statistics.median(passes)
    # the host link's floor for the same traffic: the same pipeline with the
    # compute left out (step i's inputs in while step i-1's output goes out)
    def copies(i):
        j = i % n_buf
        with torch.cuda.stream(s_in):
            for k in dev[j]:
                dev[j][k].copy_(host[j][k], non_blocking=True)
            ev["in"][j].record(s_in)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["in"][j])
            out_host[j].copy_(outs[j], non_blocking=True)
    synchronize_all(device)
    floor = []
    for _ in range(3):
        t0 = time.perf_counter()
        for i in range(steps):
            copies(i)
        synchronize_all(device)
        floor.append((time.perf_counter() - t0) / steps)
    return dt, h2d, d2h, statistics.median(floor)


def bench_decode(binding, device, steps: int, warmup: int, world: int):
    w = WORKLOADS[DECODE_WORKLOAD]
    x = inputs.workload_inputs(w, device=device)
    out = torch.empty_like(x["q"])
    ws = torch.empty(binding.decode_workspace_size(w.B, w.Hq, w.Hkv, w.S_max), dtype=torch.uint8,
                     device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        binding.decode(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                       x["start_pos"], x["q_gamma"], x["k_gamma"], w.theta, w.eps, out=out,
                       workspace=ws)

    for _ in range(warmup):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(world, device)
    synchronize_all(device)
    for i in range(steps):
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    synchronize_all(device)
    barrier(world, device)
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    status = binding.last_device_error(ws)
    if status != 0:
        raise RuntimeError(f"decode device error word: {status}")

    # the same step from a captured CUDA graph (positions in device memory)
    pos = x["start_pos"].to(device)
    graph = torch.cuda.CUDAGraph()
    synchronize_all(device)
    with torch.cuda.graph(graph):
        binding.decode_device_pos(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                                  pos, x["q_gamma"], x["k_gamma"], w.theta, w.eps, out=out,
                                  workspace=ws)
    for _ in range(warmup):
        graph.replay()
    gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    synchronize_all(device)
    for i in range(steps):
        gev[i][0].record(stream)
        graph.replay()
        gev[i][1].record(stream)
    synchronize_all(device)
    graph_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in gev)
    status = binding.last_device_error(ws)
    if status != 0:
        raise RuntimeError(f"graph decode device error word: {status}")
    return w, x["start_pos"], ms, graph_ms


def bench_chunk(binding, device, steps: int, warmup: int, world: int):
    """Chunked prefill: the caches hold each prompt's first sp_lo tokens
    (written by an untimed chunk from position 0); the timed step is the
    prompt's last T tokens as one chunk. Every step rewrites the same rows."""
    w = WORKLOADS[CHUNK_WORKLOAD]
    x = inputs.workload_inputs(w, device=device)
    p0 = w.sp_lo
    kc = torch.full((w.B, w.Hkv, w.S_max, w.d), float("nan"), dtype=torch.bfloat16, device=device)
    vc = torch.full_like(kc, float("nan"))
    head = {k: x[k][:, :p0].contiguous() for k in ("q", "k", "v")}
    tail = {k: x[k][:, p0:].contiguous() for k in ("q", "k", "v")}
    binding.prefill_chunk(head["q"], head["k"], head["v"], kc, vc, [0] * w.B, x["q_gamma"],
                          x["k_gamma"], w.theta, w.eps)
    del head
    out = torch.empty_like(tail["q"])
    ws = torch.empty(binding.prefill_chunk_workspace_size(w.B, w.T, w.Hq, w.Hkv),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    start = [p0] * w.B

    def step():
        binding.prefill_chunk(tail["q"], tail["k"], tail["v"], kc, vc, start, x["q_gamma"],
                              x["k_gamma"], w.theta, w.eps, out=out, workspace=ws)

    for _ in range(warmup):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(world, device)
    synchronize_all(device)
    for i in range(steps):
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    synchronize_all(device)
    barrier(world, device)
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    status = binding.last_device_error(ws)
    if status != 0:
        raise RuntimeError(f"chunk device error word: {status}")
    return w, start, ms


def bench_gated_chunk(binding, device, steps: int, warmup: int, world: int):
    """Gated chunked prefill: as bench_chunk, on the Qwen3-Next-shaped gated
    layer (the caches hold each prompt's first sp_lo tokens; the timed step is
    the last T tokens as one chunk)."""
    w = WORKLOADS[GATED_CHUNK_WORKLOAD]
    x = inputs.workload_inputs(w, device=device)
    p0 = w.sp_lo
    kc = torch.full((w.B, w.Hkv, w.S_max, w.d), float("nan"), dtype=torch.bfloat16, device=device)
    vc = torch.full_like(kc, float("nan"))
    head = {k: x[k][:, :p0].contiguous() for k in ("qg", "k", "v")}
    tail = {k: x[k][:, p0:].contiguous() for k in ("qg", "k", "v")}
    binding.gated_prefill_chunk(head["qg"], head["k"], head["v"], kc, vc, [0] * w.B, x["q_w"],
                                x["k_w"], w.d_r, w.theta, w.eps)
    del head
    out = torch.empty((w.B, w.T, w.Hq, w.d), dtype=torch.bfloat16, device=device)
    ws = torch.empty(binding.gated_prefill_chunk_workspace_size(w.B, w.T, w.Hq, w.Hkv),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    start = [p0] * w.B

    def step():
        binding.gated_prefill_chunk(tail["qg"], tail["k"], tail["v"], kc, vc, start, x["q_w"],
                                    x["k_w"], w.d_r, w.theta, w.eps, out=out, workspace=ws)

    for _ in range(warmup):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(world, device)
    synchronize_all(device)
    for i in range(steps):
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    synchronize_all(device)
    barrier(world, device)
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    status = binding.last_device_error(ws)
    if status != 0:
        raise RuntimeError(f"gated chunk device error word: {status}")
    return w, start, ms


def bench_gated(binding, device, steps: int, warmup: int, world: int):
    """Gated global attention of Qwen3-Next / Qwen3.5: the prologue and the
    attention kernel timed separately within each step (inputs above L2)."""
    w = WORKLOADS[GATED_WORKLOAD]
    x = inputs.workload_inputs(w, device=device)
    out = torch.empty((w.B, w.T, w.Hq, w.d), dtype=torch.bfloat16, device=device)
    ws = torch.empty(binding.gated_prefill_workspace_size(w.B, w.T, w.Hq, w.Hkv),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        binding.gated_prefill_prologue(x["qg"], x["k"], x["q_w"], x["k_w"], w.d_r, w.theta, w.eps,
                                       ws)
        if ev is not None:
            ev[1].record(stream)
        binding.gated_prefill_attention(x["qg"], x["v"], out, ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(warmup):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    barrier(world, device)
    synchronize_all(device)
    for i in range(steps):
        step(evs[i])
    synchronize_all(device)
    barrier(world, device)
    status = binding.last_device_error(ws)
    if status != 0:
        raise RuntimeError(f"gated device error word: {status}")
    pro = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    att = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    tot = statistics.mean(e[0].elapsed_time(e[2]) for e in evs)
    return w, tot, pro, att


def bench_gated_decode(binding, device, steps: int, warmup: int, world: int):
    """One gated decode step (head_dim 256, sigmoid gate) over the Qwen3-Next-shaped
    B64 caches; every step appends the same rows again."""
    w = WORKLOADS[GATED_DECODE_WORKLOAD]
    x = inputs.workload_inputs(w, device=device)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device=device)
    ws = torch.empty(binding.gated_decode_workspace_size(w.B, w.Hq, w.Hkv, w.S_max),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        binding.gated_decode(x["qg"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                             x["start_pos"], x["q_w"], x["k_w"], w.d_r, w.theta, w.eps, out=out,
                             workspace=ws)

    for _ in range(warmup):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(world, device)
    synchronize_all(device)
    for i in range(steps):
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    synchronize_all(device)
    barrier(world, device)
    status = binding.last_device_error(ws)
    if status != 0:
        raise RuntimeError(f"gated decode device error word: {status}")
    return w, x["start_pos"], statistics.mean(e[0].elapsed_time(e[1]) for e in evs)


def cpu_baseline_prefill(w, x_cpu: dict, budget_s: float = 12.0, seed: int = 0) -> dict:
    """The fp64 oracle on a bounded sample of the prefill workload's query rows
    (random (b, t, h)), on all host cores, for about ``budget_s`` seconds."""
    import oracle

    oracle.build()
    g = torch.Generator().manual_seed(seed)
    rows_done, flops = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        n = 16
        rows = torch.stack([torch.randint(0, w.B, (n,), generator=g),
                            torch.randint(0, w.T, (n,), generator=g),
                            torch.randint(0, w.Hq, (n,), generator=g)], 1).to(torch.int32)
        oracle.prefill_rows(x_cpu["q"], x_cpu["k"], x_cpu["v"], x_cpu["q_gamma"],
                            x_cpu["k_gamma"], w.theta, w.eps, rows)
        rows_done += n
        flops += sum(4 * w.d * (int(t) + 1) for t in rows[:, 1].tolist())
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": f"{rows_done} random query rows (b,t,h) of {w.name}, each computed from "
                      f"scratch in fp64 (its keys normalised and rotated again); {dt:.1f} s wall"}


def run_profile_case(which: str) -> None:
    """A few launches of one kernel on a case sized for an ncu capture
    (inputs larger than L2, a few GB on the device at most)."""
    from qwen3_qk_norm_gb300 import binding
    from qwen3_qk_norm_gb300.build import build
    build()
    device = torch.device("cuda", 0)
    if which == "prefill":
        w = WORKLOADS[PREFILL_WORKLOAD]
        x = inputs.workload_inputs(w, device=device)
        for _ in range(3):
            binding.prefill(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], w.theta, w.eps)
    elif which == "chunk":
        bench_chunk(binding, device, 3, 0, 1)
    elif which == "gated":
        bench_gated(binding, device, 3, 0, 1)
    elif which == "gated_chunk":
        bench_gated_chunk(binding, device, 3, 0, 1)
    elif which == "gated_decode":
        w = WORKLOADS[GATED_DECODE_WORKLOAD]
        B = 16  # a quarter of the batch: about 1 GB of cache
        x = inputs.gated_decode_inputs(B, w.Hq, w.Hkv, w.S_max, w.sp_lo, w.sp_hi, w.d, w.seed,
                                       device=device)
        for _ in range(3):
            binding.gated_decode(x["qg"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                                 x["start_pos"], x["q_w"], x["k_w"], w.d_r, w.theta, w.eps)
        print(json.dumps({"gated_decode_bytes_per_step": accounting.gated_decode_bytes(
            x["start_pos"].tolist(), w.Hq, w.Hkv, w.d), "B": B}))
    else:
        w = WORKLOADS[DECODE_WORKLOAD]
        B = 16  # a quarter of the batch: 2 GiB of cache instead of 8
        x = inputs.decode_inputs(B, w.Hq, w.Hkv, w.S_max, w.sp_lo, w.sp_hi, w.d, w.seed,
                                 device=device)
        for _ in range(3):
            binding.decode(x["q"], x["k_new"], x["v_new"], x["k_cache"], x["v_cache"],
                           x["start_pos"], x["q_gamma"], x["k_gamma"], w.theta, w.eps)
        print(json.dumps({"decode_bytes_per_step": accounting.decode_bytes(
            x["start_pos"].tolist(), w.Hq, w.Hkv, w.d), "B": B}))
    torch.cuda.synchronize(device)


def run_ours(args) -> None:
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    from qwen3_qk_norm_gb300 import binding
    from qwen3_qk_norm_gb300.build import build
    build()
    binding.load()
    peaks, peak_src = measured_peaks()

    with ClockSampler(device) as clk:
        w, x, step_ms, k1_ms, k2_ms = bench_prefill(binding, device, args.steps, args.warmup, world,
                                                    args.prefill_workload)
        dw, start_pos, dec_ms, dec_graph_ms = (None, None, None, None)
        if not args.no_decode:
            dw, start_pos, dec_ms, dec_graph_ms = bench_decode(binding, device, args.steps,
                                                               args.warmup, world)
        cw, c_start, ch_ms = (None, None, None)
        if not args.no_chunk:
            cw, c_start, ch_ms = bench_chunk(binding, device, args.steps, args.warmup, world)
        gw, g_ms, gp_ms, ga_ms = (None, None, None, None)
        gdw, gd_start, gd_ms = (None, None, None)
        gcw, gc_start, gc_ms = (None, None, None)
        if not args.no_gated:
            gw, g_ms, gp_ms, ga_ms = bench_gated(binding, device, args.steps, args.warmup, world)
            gdw, gd_start, gd_ms = bench_gated_decode(binding, device, args.steps, args.warmup,
                                                      world)
            if not args.no_chunk:
                gcw, gc_start, gc_ms = bench_gated_chunk(binding, device, args.steps, args.warmup,
                                                         world)
    clocks = clk.summary()

    flops = accounting.prefill_flops(w.B, w.T, w.Hq, w.d)
    step_ms_max = max_over_ranks(step_ms, world, device)
    k2_ms_max = max_over_ranks(k2_ms, world, device)
    k1_ms_max = max_over_ranks(k1_ms, world, device)
    value = whole_job_rate(flops, world, step_ms_max / 1e3) / 1e12
    k2_tflops = flops / (k2_ms_max / 1e3) / 1e12
    # the prologue normalises the keys (read + write) and writes the table of
    # RoPE cos/sin per position; the query tiles are normalised inside K2
    k1_bytes = (w.B * w.T * w.Hkv * w.d * 2) * 2 + w.T * 64 * 8 + 2 * w.d * 2
    traffic = ncu_traffic("prefill_attention_kernel")

    # the other prefill workloads, each timed as the headline one (K1 and K2 by
    # events within every step)
    extra = {}
    if not args.no_prefill_configs:
        with ClockSampler(device) as clk2:
            for name in EXTRA_PREFILL_WORKLOADS:
                if name == w.name:
                    continue
                ew, ex, e_step, e_k1, e_k2 = bench_prefill(binding, device, args.steps,
                                                           args.warmup, world, name)
                del ex
                torch.cuda.empty_cache()
                extra[name] = (ew, max_over_ranks(e_step, world, device),
                               max_over_ranks(e_k1, world, device),
                               max_over_ranks(e_k2, world, device))
        extra_clocks = clk2.summary()

    e2e_steps = max(1, min(args.steps, 10))
    e2e_dt, h2d, d2h, e2e_floor = bench_prefill_e2e(binding, device, w, e2e_steps)
    e2e_dt = max_over_ranks(e2e_dt, world, device)

    step_bytes = w.B * w.T * (3 * w.Hq + 3 * w.Hkv) * w.d * 2
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                   "theta": w.theta, "eps": w.eps, "outliers": (f"{w.outlier_frac:.0%} of Q/K rows x{w.outlier_scale:g}"
                                 if w.outlier_frac > 0 else "none"),
                   "causal": True, "parallelism": f"replicas x{world} (weak, no collective)",
                   "l2": (f"inputs {'larger' if step_bytes > L2_BYTES else 'SMALLER'} than L2 "
                          f"(no flush): q,k,v,Qhat,Khat,out = {step_bytes / 2**20:.0f} MiB "
                          "per step")},
        "roofline": {"bound": "tensor", "kernel": "prefill_attention_kernel",
                     "achieved": round(k2_tflops, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(k2_tflops / peaks["bf16_tflops"], 4),
                     "peak_source": f"{peak_src} bf16 dense burst",
                     "frac_of_sustained": round(k2_tflops / peaks.get(
                         "bf16_tflops_sustained", peaks["bf16_tflops"]), 4),
                     "traffic": traffic, "flops_per_launch": flops,
                     "ms_per_launch": round(k2_ms_max, 4)},
        "prologue": {"kernel": "qknorm_rope_kernel", "ms_per_launch": round(k1_ms_max, 4),
                     "bytes_per_launch": k1_bytes,
                     "achieved_gbs": round(k1_bytes / (k1_ms_max / 1e3) / 1e9, 1),
                     "frac_of_hbm": round(k1_bytes / (k1_ms_max / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                     "traffic": ncu_traffic("qknorm_rope_kernel")},
        "e2e": {"value": round(whole_job_rate(flops, world, e2e_dt) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "q3a_prefill with pinned host inputs copied in and the output copied out "
                       "every step; copy-in, compute and copy-out on three streams with two "
                       "buffer sets, so step i+1's inputs travel while step i computes; median "
                       "of three timed passes of up to 10 steps after 3 warm-up steps",
                "ms_per_step": round(e2e_dt * 1e3, 4),
                # the same copies with the compute left out: the host link's floor
                "copy_only_ms_per_step": round(e2e_floor * 1e3, 4),
                "frac_of_copy_floor": round(e2e_floor / e2e_dt, 3) if e2e_dt > 0 else None},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    line["step_frac_of_peak"] = round(value / world / peaks["bf16_tflops"], 4)
    if extra:
        cfgs = {}
        for name, (ew, e_step, e_k1, e_k2) in extra.items():
            ef = accounting.prefill_flops(ew.B, ew.T, ew.Hq, ew.d)
            e_bytes = ew.B * ew.T * (3 * ew.Hq + 3 * ew.Hkv) * ew.d * 2
            k2_rate = ef / (e_k2 / 1e3) / 1e12
            cfgs[name] = {
                "value": round(whole_job_rate(ef, world, e_step / 1e3) / 1e12, 2),
                "unit": "TFLOP/s", "ms_per_step": round(e_step, 4),
                "us_per_step": round(e_step * 1e3, 1),
                "step_frac_of_peak": round(ef / (e_step / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
                "config": {"B": ew.B, "T": ew.T, "Hq": ew.Hq, "Hkv": ew.Hkv, "d": ew.d,
                           "theta": ew.theta, "flops_per_step": ef,
                           "l2": (f"inputs {'larger' if e_bytes > L2_BYTES else 'SMALLER'} than L2"
                                  f" (no flush): {e_bytes / 2**20:.1f} MiB per step")},
                "roofline": {"bound": "tensor", "kernel": "prefill_attention_kernel",
                             "achieved": round(k2_rate, 2), "peak": peaks["bf16_tflops"],
                             "unit": "TFLOP/s", "frac": round(k2_rate / peaks["bf16_tflops"], 4),
                             "peak_source": f"{peak_src} bf16 dense burst",
                             "frac_of_sustained": round(k2_rate / peaks.get(
                                 "bf16_tflops_sustained", peaks["bf16_tflops"]), 4),
                             "ms_per_launch": round(e_k2, 4)},
                "prologue_ms_per_launch": round(e_k1, 4),
                "gpu_launches": 2 * args.steps,
            }
        line["prefill_configs"] = {"workloads": cfgs, "clocks": extra_clocks,
                                   "api": "q3a_prefill_prologue + q3a_prefill_attention, "
                                          "timed as the headline step"}
    if dec_ms is not None:
        dbytes = accounting.decode_bytes(start_pos.tolist(), dw.Hq, dw.Hkv, dw.d)
        dec_ms_max = max_over_ranks(dec_ms, world, device)
        gbs = whole_job_rate(dbytes, world, dec_ms_max / 1e3) / 1e9
        per_gpu = dbytes / (dec_ms_max / 1e3) / 1e9
        line["decode"] = {
            "value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(dec_ms_max, 4),
            "config": {"workload": dw.name, "B": dw.B, "Hq": dw.Hq, "Hkv": dw.Hkv,
                       "S_max": dw.S_max, "start_pos": f"U[{dw.sp_lo}, {dw.sp_hi}) seed {dw.seed}",
                       "bytes_per_step": dbytes},
            "roofline": {"bound": "hbm", "kernel": "decode_split_kernel + decode_combine_kernel",
                         "achieved": round(per_gpu, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(per_gpu / peaks["hbm_gbs"], 4),
                         "peak_source": f"{peak_src} copy bandwidth",
                         "traffic": ncu_traffic("decode_split_kernel")},
            "gpu_launches": 2 * args.steps,
            "graph": {"api": "q3a_decode_device_pos captured in a CUDA graph, replayed",
                      "ms_per_step": round(dec_graph_ms, 4),
                      "value": round(dbytes / (dec_graph_ms / 1e3) / 1e9, 1), "unit": "GB/s",
                      "gpu_launches": 3 * args.steps},
        }
    if ch_ms is not None:
        cflops = accounting.chunk_flops(c_start, cw.T, cw.Hq, cw.d)
        ch_ms_max = max_over_ranks(ch_ms, world, device)
        per_gpu = cflops / (ch_ms_max / 1e3) / 1e12
        line["chunk"] = {
            "value": round(whole_job_rate(cflops, world, ch_ms_max / 1e3) / 1e12, 2),
            "unit": "TFLOP/s", "ms_per_step": round(ch_ms_max, 4),
            "config": {"workload": cw.name, "B": cw.B, "Tq": cw.T, "start_pos": cw.sp_lo,
                       "Hq": cw.Hq, "Hkv": cw.Hkv, "S_max": cw.S_max, "flops_per_step": cflops,
                       "api": "q3a_prefill_chunk (prologue writes the chunk into the caches, "
                              "attention reads them)"},
            "roofline": {"bound": "tensor", "kernel": "qknorm_rope_kernel + "
                         "prefill_attention_kernel<PrefillChunkArgs>",
                         "achieved": round(per_gpu, 2), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(per_gpu / peaks["bf16_tflops"], 4),
                         "peak_source": f"{peak_src} bf16 dense burst",
                         "traffic": ncu_traffic("prefill_attention_kernel<chunk>")},
            "gpu_launches": 2 * args.steps,
        }
    if g_ms is not None:
        gflops = accounting.prefill_flops(gw.B, gw.T, gw.Hq, gw.d)
        g_max, ga_max, gp_max = (max_over_ranks(v, world, device) for v in (g_ms, ga_ms, gp_ms))
        att = gflops / (ga_max / 1e3) / 1e12
        gp_bytes = 2 * gw.B * gw.T * (gw.Hq + gw.Hkv) * gw.d * 2 + 2 * gw.d * 2
        line["gated"] = {
            "value": round(whole_job_rate(gflops, world, g_max / 1e3) / 1e12, 2),
            "unit": "TFLOP/s", "ms_per_step": round(g_max, 4),
            "config": {"workload": gw.name, "B": gw.B, "T": gw.T, "Hq": gw.Hq, "Hkv": gw.Hkv,
                       "d": gw.d, "d_rot": gw.d_r, "theta": gw.theta, "flops_per_step": gflops,
                       "api": "q3a_gated_prefill_prologue + q3a_gated_prefill_attention"},
            "roofline": {"bound": "tensor", "kernel": "gated_attention_pair_kernel",
                         "achieved": round(att, 2), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(att / peaks["bf16_tflops"], 4),
                         "peak_source": f"{peak_src} bf16 dense burst",
                         "traffic": ncu_traffic("gated_attention_pair_kernel"),
                         "ms_per_launch": round(ga_max, 4)},
            "prologue": {"kernel": "gated_prologue_kernel", "ms_per_launch": round(gp_max, 4),
                         "bytes_per_launch": gp_bytes,
                         "achieved_gbs": round(gp_bytes / (gp_max / 1e3) / 1e9, 1),
                         "frac_of_hbm": round(gp_bytes / (gp_max / 1e3) / 1e9 / peaks["hbm_gbs"],
                                              4),
                         "traffic": ncu_traffic("gated_prologue_kernel")},
            "gpu_launches": 2 * args.steps,
        }
    if gd_ms is not None:
        gbytes = accounting.gated_decode_bytes(gd_start.tolist(), gdw.Hq, gdw.Hkv, gdw.d)
        gd_max = max_over_ranks(gd_ms, world, device)
        per_gpu = gbytes / (gd_max / 1e3) / 1e9
        line["gated_decode"] = {
            "value": round(whole_job_rate(gbytes, world, gd_max / 1e3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(gd_max, 4),
            "config": {"workload": gdw.name, "B": gdw.B, "Hq": gdw.Hq, "Hkv": gdw.Hkv, "d": gdw.d,
                       "d_rot": gdw.d_r, "S_max": gdw.S_max,
                       "start_pos": f"U[{gdw.sp_lo}, {gdw.sp_hi}) seed {gdw.seed}",
                       "bytes_per_step": gbytes, "api": "q3a_gated_decode"},
            "roofline": {"bound": "hbm", "kernel": "decode_split_kernel<256> + "
                         "decode_combine_kernel<256>",
                         "achieved": round(per_gpu, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(per_gpu / peaks["hbm_gbs"], 4),
                         "peak_source": f"{peak_src} copy bandwidth",
                         "traffic": ncu_traffic("decode_split_kernel<256>")},
            "gpu_launches": 2 * args.steps,
        }
    if gc_ms is not None:
        cflops = accounting.chunk_flops(gc_start, gcw.T, gcw.Hq, gcw.d)
        gc_max = max_over_ranks(gc_ms, world, device)
        per_gpu = cflops / (gc_max / 1e3) / 1e12
        line["gated_chunk"] = {
            "value": round(whole_job_rate(cflops, world, gc_max / 1e3) / 1e12, 2),
            "unit": "TFLOP/s", "ms_per_step": round(gc_max, 4),
            "config": {"workload": gcw.name, "B": gcw.B, "Tq": gcw.T, "start_pos": gcw.sp_lo,
                       "Hq": gcw.Hq, "Hkv": gcw.Hkv, "d": gcw.d, "d_rot": gcw.d_r,
                       "S_max": gcw.S_max, "flops_per_step": cflops,
                       "api": "q3a_gated_prefill_chunk (prologue writes the chunk into the "
                              "caches, attention reads them)"},
            "roofline": {"bound": "tensor", "kernel": "gated_prologue_kernel<chunk> + "
                         "gated_attention_pair_kernel<GatedAttnChunkArgs>",
                         "achieved": round(per_gpu, 2), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(per_gpu / peaks["bf16_tflops"], 4),
                         "peak_source": f"{peak_src} bf16 dense burst",
                         "traffic": ncu_traffic("gated_attention_pair_kernel<chunk>")},
            "gpu_launches": 2 * args.steps,
        }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x_cpu = {k: t.cpu() for k, t in x.items()}
        line["cpu_baseline"] = cpu_baseline_prefill(w, x_cpu)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle on bounded samples of the same workload
# ----------------------------------------------------------------------------
def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    w = WORKLOADS[PREFILL_WORKLOAD]
    x = inputs.workload_inputs(w, device="cpu")
    g = torch.Generator().manual_seed(1234)
    n_rows = 8

    def one_step():
        rows = torch.stack([torch.randint(0, w.B, (n_rows,), generator=g),
                            torch.randint(0, w.T, (n_rows,), generator=g),
                            torch.randint(0, w.Hq, (n_rows,), generator=g)], 1).to(torch.int32)
        t0 = time.perf_counter()
        oracle.prefill_rows(x["q"], x["k"], x["v"], x["q_gamma"], x["k_gamma"], w.theta, w.eps,
                            rows)
        return time.perf_counter() - t0, sum(4 * w.d * (int(t) + 1) for t in rows[:, 1].tolist())

    for _ in range(args.warmup):
        one_step()
    secs, flops = 0.0, 0
    for _ in range(args.steps):
        s, f = one_step()
        secs += s
        flops += f
    value = flops / secs / 1e12
    sample = f"{n_rows} random query rows of {w.name} per step, fp64, each row from scratch"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-chunk", action="store_true")
    ap.add_argument("--no-gated", action="store_true")
    ap.add_argument("--no-prefill-configs", action="store_true",
                    help="skip the other prefill workloads (tiny, 32B-shaped, 30B-A3B-shaped)")
    ap.add_argument("--prefill-workload", default=PREFILL_WORKLOAD,
                    choices=[n for n, w in WORKLOADS.items() if w.kind == "prefill"],
                    help="prefill workload of the step (the default is the headline one)")
    ap.add_argument("--profile-case",
                    choices=["prefill", "decode", "chunk", "gated", "gated_decode",
                             "gated_chunk"],
                    help="run a few launches of one kernel for an ncu capture, print no JSON")
    args = ap.parse_args(argv)
    if args.profile_case:
        run_profile_case(args.profile_case)
        return
    if args.warmup < 3:
        args.warmup = 3  # never time cold kernels
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
