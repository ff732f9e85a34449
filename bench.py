"""Benchmark of the preshuffle GEMM on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--no-others]

One step is one gemm_run call (C = A . B^T with B already packed) on the
named workload: the hot path with the weight resident in HBM.  The offline
preshuffle of B is timed separately (key "pack_b") because the method runs
it once per weight, not per product.

- L2: each step uses its own packed-B / A copy, rotating through enough
  copies that their total exceeds 2x the 129 MB L2.  Every step therefore
  streams B from HBM.
- Timing: W warm-up steps, then exactly K steps, replayed from a CUDA graph
  of back-to-back gemm_run launches (no host gaps).  The K steps sit between
  a barrier and torch.cuda.synchronize() on both sides and are timed with
  CUDA events on the launch stream; a short device spin queued ahead of the
  start event keeps the host's graph submission out of the device time.
- Reported value: the maximum over ranks.  Under torchrun every rank runs the
  same independent problem on its own GPU (weak scaling, no collective).
- JSON line keys:
  - "e2e": the same metric through the public call, with pinned host
    buffers.  A and its scales are copied host->device and C device->host
    every step; successive steps alternate over 16 streams (independent
    requests), so the copies of one step overlap the GEMM of another, and
    the steps are replayed from CUDA graphs (copies included), as a serving
    loop would.
  - "roofline": the GEMM kernel against the measured HBM or tensor peak.
  - "tensor_rates": this GPU's tcgen05 MMA rate per kind (a loop with no
    memory traffic, rates/mma_rate.cu in the package) and its ratio to
    bf16; tensor rooflines add "frac_of_measured_ratio_peak", the measured
    bf16 peak times that ratio, beside "frac" (the nominal ratio).
  - "cpu_baseline": the oracle, timed on this host's cores on a bounded
    sample; "cpu_oracle_others": the same for each other workload (a
    shorter sample each).
  - "others": the other workloads, each with its own device-timed TFLOP/s
    and roofline fraction.
  - "epilogues": each float workload with the fused bias + GELU epilogue,
    beside the plain product's time.
  - "quantize": the activation quantiser (gemm_quantize_a) on the FP8 and
    MXFP4 workloads' A shapes, against the HBM roofline.
  - "trials" (in the line and each "others" entry): 7 trials of 80
    back-to-back steps; median, p10 and p90 of the time per step.
  - "independent_stream": the INT8 and W4A8 workloads as runs of calls with
    GP_RUN_INDEPENDENT (each on its own weights and output).
  - "b_default": the headline workload through plain gemm_run (no flag).
  - "a_l2_resident": the headline workload with one A buffer for every step
    (L2-resident, as the previous kernel's output would be), B still
    rotating past L2; the headline itself keeps a fresh A copy per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from typing import Optional

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS & % of GB300 dtype peak; HBM GB/s % for small-M shapes"
DEFAULT_WORKLOAD = "int8_16x7168x4096"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal dense tensor-rate ratios to bf16 (2.25 PF): fp8 4.5, fp4 13.5
DTYPE_RATIO = {"bf16": 1.0, "fp16": 1.0, "e4m3": 2.0, "e2m1": 6.0}
B_DEFAULT_FLAGS = False  # --b-default: time gemm_run without GP_RUN_B_CONSTANT
# tcgen05 MMA rates of this GPU by kind (rates/mma_rate.cu), measured once per
# run on rank 0: the ratios of FP8 and MXFP4 to bf16 beside the nominal ones
MMA_RATES = None
HOST_COVER_CYCLES = 200_000  # ~0.1 ms of device spin before a timed region (see time_device)


def tensor_rates():
    """Run the library's tensor-pipe rate probe (built beside it by build()):
    TFLOP/s of back-to-back MMAs of each kind with no memory traffic, in the
    single-CTA and the 2-CTA (pair) form.  Returns {kind: TFLOP/s} (the
    higher of the two forms), the ratio of each kind to bf16, and the lines
    it printed; None if the probe is missing or fails."""
    import subprocess
    exe = os.path.join(ROOT, "dense_gemm_preshuffle_gb300", "_lib", "mma_rate")
    if not os.path.exists(exe):
        return None
    try:
        r = subprocess.run([exe, "20000", "1"], capture_output=True, text=True, timeout=120)
    except (OSError, subprocess.TimeoutExpired):
        return None
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    best = {}
    for d in lines:
        if d.get("ok") and "tflops" in d:
            best[d["kind"]] = max(best.get(d["kind"], 0.0), d["tflops"])
    if r.returncode != 0 or "bf16" not in best:
        return None
    return {"tflops": best, "ratio_to_bf16": {k: round(v / best["bf16"], 3) for k, v in best.items()},
            "runs": lines, "source": "dense_gemm_preshuffle_gb300/rates/mma_rate.cu, 20000 loops, this run"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_bytes(dtype: str, M: int, N: int, K: int) -> int:
    """A + B + C + scales, as the GEMM guide counts them (section 8.2); the
    INT8 workload's C is int32 and it has no scales."""
    if dtype == "int8":
        return M * K + N * K + M * N * 4
    if dtype == "w4a8":
        return M * K + N * K // 2 + M * N * 4
    if dtype == "e4m3":
        return M * K + N * K + M * N * 2 + (M + N) * 4
    if dtype in ("bf16", "fp16"):
        return 2 * M * K + 2 * N * K + 2 * M * N
    if dtype == "e2m1":
        return M * K // 2 + N * K // 2 + M * N * 2 + (M + N) * (K // 32)
    raise ValueError(dtype)


def workload_config(name: str, M: int, N: int, K: int) -> dict:
    """The JSON line's `config`, the same keys in both arms."""
    return {"workload": name, "M": M, "N": N, "K": K}


def bound_of(dtype: str, M: int) -> str:
    # the guide's rule of thumb (section 8.3): M <= 512 memory-bound; the
    # int8 small-batch workload is the weight-streaming case
    return "hbm" if dtype in ("int8", "w4a8") else "tensor"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.perf_counter(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        use = inside if inside else [p for (t, p) in self.samples]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in use if num(p[0]) is not None]
        mx = [num(p[1]) for p in use if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4) if p[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside),
                "power_w_max": max((num(p[2]) or 0.0) for p in use)}


# ------------------------------------------------------------------ distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device])
        else:
            pg.barrier()


def max_over_ranks(pg, x: float, device=None):
    """The maximum of x over all ranks (x itself without a process group)."""
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world: int, flops_per_step: float, steps: int, max_seconds: float) -> float:
    """Weak scaling: every rank runs its own problem; the job's throughput is
    all ranks' work over the slowest rank's time (TFLOP/s)."""
    return world * flops_per_step * steps / max_seconds / 1e12


# ------------------------------------------------------------------ our arm

class Problem:
    """Device-resident copies of one workload, ready for gemm_run."""

    def __init__(self, name: str, device, copies: int | None = None):
        import torch
        import dense_gemm_preshuffle_gb300 as gp
        from dense_gemm_preshuffle_gb300 import inputs
        self.gp = gp
        self.name = name
        self.ops = ops = inputs.workload_operands(name)
        self.dtype, self.M, self.N, self.K = ops.dtype, ops.M, ops.N, ops.K

        def t(x):
            if x is None:
                return None
            if x.dtype == np.uint16:
                x = x.view(np.int16)
            return torch.from_numpy(np.ascontiguousarray(x))
        self.host_a, self.host_sa = t(ops.a), t(ops.scale_a)
        B = t(ops.b).to(device)
        sb = t(ops.scale_b).to(device) if ops.scale_b is not None else None
        # time the offline pack on the device (a CUDA graph of pack calls over
        # copies of B that rotate past L2), then pack once for the GEMM
        bsf = sb if self.dtype == "e2m1" else None
        pack = PackProblem(gp, self.dtype, self.N, self.K, B, bsf, device)
        pack_steps = max(20, pack.copies)
        self.pack_us = time_device(pack, pack_steps, 3, None, device) / pack_steps * 1e6
        del pack
        bp = torch.empty(gp.gemm_packed_b_bytes(self.dtype, self.N, self.K), dtype=torch.uint8, device=device)
        gp.gemm_preshuffle_b(B, bsf, self.dtype, self.N, self.K, bp)
        torch.cuda.synchronize(device)
        self.packed_bytes = bp.numel()
        if copies is None:
            copies = max(1, math.ceil(2 * L2_BYTES / max(1, bp.numel())) + 1)
        self.copies = copies
        self.Bp = [bp] + [bp.clone() for _ in range(copies - 1)]
        A = self.host_a.to(device)
        self.A = [A] + [A.clone() for _ in range(copies - 1)]
        self.sa = self.host_sa.to(device) if self.host_sa is not None else None
        self.sb = sb if self.dtype == "e4m3" else None
        cdt = torch.int32 if self.dtype in ("int8", "w4a8") else (
            torch.float16 if self.dtype == "fp16" else torch.bfloat16)
        # one output per copy when small (independent calls write outputs of their own)
        c_bytes = self.M * self.N * (4 if cdt == torch.int32 else 2)
        n_c = copies if c_bytes <= (64 << 20) else min(copies, 4)
        self.C = [torch.empty((self.M, self.N), dtype=cdt, device=device) for _ in range(n_c)]
        self.c_dtype = {"int8": "int32", "w4a8": "int32", "fp16": "fp16"}.get(self.dtype, "bf16")
        self.mode = {"int8": "none", "w4a8": "none", "bf16": "none", "fp16": "none", "e4m3": "rowcol_f32",
                     "e2m1": "block32_ue8m0"}[self.dtype]
        self.flops = 2 * self.M * self.N * self.K
        self.bytes = algorithmic_bytes(self.dtype, self.M, self.N, self.K)
        # the packed weights are complete (synchronised above) and never
        # rewritten: every step may pass GP_RUN_B_CONSTANT
        self.flags = gp.GP_RUN_DEFAULT if B_DEFAULT_FLAGS else gp.GP_RUN_B_CONSTANT
        self.epilogue, self.bias = "none", None

    def step(self, i: int, stream=None):
        j = i % self.copies
        self.gp.gemm_run_ex(self.A[j], self.Bp[j], self.dtype, self.M, self.N, self.K, self.mode,
                            self.sa, self.sb, self.epilogue, self.bias, self.C[j % len(self.C)], self.c_dtype,
                            self.flags, stream)


def gpu_record(device) -> dict:
    """The GPU the numbers were taken on (name, SMs, L2, compute capability)."""
    import torch
    pr = torch.cuda.get_device_properties(device)
    return {"name": pr.name, "sms": pr.multi_processor_count, "l2_bytes": getattr(pr, "L2_cache_size", None),
            "cc": f"{pr.major}.{pr.minor}", "memory_bytes": pr.total_memory}


class PackProblem:
    """The offline pack of B as a timed step: copies of B (and of the packed
    output) rotate past L2, so each pack reads and writes HBM."""

    def __init__(self, gp, dtype, N, K, B, bsf, device):
        import torch
        self.gp, self.dtype, self.N, self.K, self.bsf = gp, dtype, N, K, bsf
        out_bytes = gp.gemm_packed_b_bytes(dtype, N, K)
        pair = B.numel() * B.element_size() + out_bytes
        self.copies = max(1, math.ceil(2 * L2_BYTES / max(1, pair)) + 1)
        self.B = [B] + [B.clone() for _ in range(self.copies - 1)]
        self.out = [torch.empty(out_bytes, dtype=torch.uint8, device=device) for _ in range(self.copies)]

    def step(self, i: int, stream=None):
        j = i % self.copies
        self.gp.gemm_preshuffle_b(self.B[j], self.bsf, self.dtype, self.N, self.K, self.out[j], stream)


def time_device(prob: Problem, steps: int, warmup: int, pg, device, graph_len: int = 100):
    """Device time (s) of exactly `steps` steps after `warmup` warm-up steps."""
    import torch
    stream = torch.cuda.current_stream(device)
    for i in range(max(3, warmup)):
        prob.step(i)
    torch.cuda.synchronize(device)
    # the graph covers every rotating copy (else a small workload's replays
    # would cycle through only graph_len copies, which stay in L2)
    g_len = max(1, min(steps, max(graph_len, prob.copies)))
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for i in range(g_len):
                prob.step(i)
    stream.wait_stream(s)
    graph.replay()  # untimed warm replay
    torch.cuda.synchronize(device)
    full, rest = divmod(steps, g_len)
    tail = None
    if rest:
        # the last `rest` steps as a graph of their own (no host gaps)
        tail = torch.cuda.CUDAGraph()
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            with torch.cuda.graph(tail, stream=s):
                for i in range(rest):
                    prob.step(i)
        stream.wait_stream(s)
        tail.replay()
        torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg, device.index if pg is not None else None)
    torch.cuda.synchronize(device)
    # A short device spin ahead of the start event: the event is then taken
    # once the host has submitted the graph, so the host's submission latency
    # is not counted as device time (it would be ~10 us in a 20-step run).
    torch.cuda._sleep(HOST_COVER_CYCLES)
    e0.record(stream)
    for _ in range(full):
        graph.replay()
    if tail is not None:
        tail.replay()
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(pg, device.index if pg is not None else None)
    return e0.elapsed_time(e1) / 1e3


def time_trials(prob, warmup: int, device, R: int = 80, n: int = 7):
    """n trials of R back-to-back steps (one CUDA-graph replay each): the
    median, p10 and p90 of the per-step device time, in microseconds.  R is
    raised to the number of rotating copies, so a trial's inputs exceed L2."""
    import torch
    R = max(R, prob.copies)
    stream = torch.cuda.current_stream(device)
    for i in range(max(3, warmup)):
        prob.step(i)
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for i in range(R):
                prob.step(i)
    stream.wait_stream(s)
    graph.replay()
    torch.cuda.synchronize(device)
    per = []
    for _ in range(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(HOST_COVER_CYCLES)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(device)
        per.append(e0.elapsed_time(e1) * 1e3 / R)
    q = np.percentile(np.array(per), [10, 50, 90])
    return {"R": R, "n": n, "median_us": round(float(q[1]), 3), "p10_us": round(float(q[0]), 3),
            "p90_us": round(float(q[2]), 3)}


class QuantProblem:
    """gemm_quantize_a on an activation matrix [M, K] (rotating copies past L2)."""

    def __init__(self, q: str, xd: str, M: int, K: int, device):
        import torch
        import dense_gemm_preshuffle_gb300 as gp
        self.gp, self.q, self.xd, self.M, self.K = gp, q, xd, M, K
        tdt = torch.bfloat16 if xd == "bf16" else torch.float32
        x = torch.randn((M, K), generator=torch.Generator().manual_seed(5), dtype=torch.float32).to(tdt).to(device)
        xbytes = x.numel() * x.element_size()
        self.copies = max(1, math.ceil(2 * L2_BYTES / xbytes) + 1)
        self.X = [x] + [x.clone() for _ in range(self.copies - 1)]
        self.A, self.S = gp.quantize(x, q)
        code_bytes = M * K if q == "e4m3" else M * K // 2
        scale_bytes = M * 4 if q == "e4m3" else M * K // 32
        self.bytes = xbytes + code_bytes + scale_bytes

    def step(self, i: int, stream=None):
        self.gp.gemm_quantize_a(self.X[i % self.copies], self.xd, self.M, self.K, self.q, self.A, self.S, stream)


def time_quantizers(args, pg, device, peaks, peak_kind):
    """The activation quantiser on the FP8 and MXFP4 workloads' A shapes, from
    fp32 and bf16: device time against the HBM roofline (read x, write codes
    and scales)."""
    import torch
    res = {}
    for q, M, K in (("e4m3", 8192, 8192), ("e2m1", 4096, 8192)):
        for xd in ("fp32", "bf16"):
            name = f"{q}_{M}x{K}_from_{xd}"
            try:
                p = QuantProblem(q, xd, M, K, device)
                steps = max(20, min(args.steps, 400), p.copies)
                sec = max_over_ranks(pg, time_device(p, steps, args.warmup, pg, device), device)
                per = sec / steps
                achieved = p.bytes / per / 1e9
                peak = peaks["hbm_gbs"]
                res[name] = {"us_per_call": round(per * 1e6, 3), "GB/s": round(achieved, 1),
                             "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                                          "unit": "GB/s", "frac": round(achieved / peak, 4),
                                          "traffic": traffic_from_profiles("quantize_" + name),
                                          "algorithmic_bytes_per_launch": p.bytes,
                                          "peak_source": f"hbm_gbs ({peak_kind})"}}
                del p
                torch.cuda.empty_cache()
            except Exception as e:
                res[name] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
    return res


# streams the end-to-end steps alternate over (BENCH_E2E_STREAMS overrides)
E2E_STREAMS = int(os.environ.get("BENCH_E2E_STREAMS", "16"))


def time_e2e(prob: Problem, steps: int, warmup: int, device, record: Optional[dict] = None):
    """Through the public call with pinned host buffers: H2D of A (+ its
    scales), gemm_run_ex, D2H of C, every step.  Successive steps alternate
    over E2E_STREAMS streams, so one step's copies overlap another's GEMM
    (each device and host buffer is only ever used by steps of one stream,
    so stream order alone keeps the buffers consistent).  Returns (seconds,
    h2d bytes, d2h bytes) per step.  `record`, if given, receives the device
    and host output buffers (for the tests)."""
    import torch
    S = E2E_STREAMS
    ha = prob.host_a.pin_memory()
    hsa = prob.host_sa.pin_memory() if prob.host_sa is not None else None
    hc = [torch.empty(prob.C[0].shape, dtype=prob.C[0].dtype).pin_memory() for _ in range(S)]
    # per-stream device scales (the row scales are an input of every step)
    sa = [prob.sa.clone() if prob.sa is not None else None for _ in range(S)]
    nA = max(S, (prob.copies // S) * S)
    nC = max(S, (len(prob.C) // S) * S)
    A = [prob.A[k % len(prob.A)] if k < len(prob.A) else prob.A[0].clone() for k in range(nA)]
    C = [prob.C[k] if k < len(prob.C) else torch.empty_like(prob.C[0]) for k in range(nC)]
    main = torch.cuda.current_stream(device)
    streams = [torch.cuda.Stream(device) for _ in range(S)]

    def one(i):
        s = i % S
        st = streams[s]
        with torch.cuda.stream(st):
            a = A[i % nA]            # i % nA has the parity of i: only stream s uses it
            c = C[i % nC]
            a.copy_(ha, non_blocking=True)
            if hsa is not None:
                sa[s].copy_(hsa, non_blocking=True)
            prob.gp.gemm_run_ex(a, prob.Bp[i % prob.copies], prob.dtype, prob.M, prob.N, prob.K, prob.mode, sa[s],
                                prob.sb, prob.epilogue, prob.bias, c, prob.c_dtype, prob.flags, st)
            hc[s].copy_(c, non_blocking=True)

    for st in streams:
        st.wait_stream(main)
    for i in range(max(3, warmup)):
        one(i)
    torch.cuda.synchronize(device)
    # Serving replays captured steps (the copies are graph memcpy nodes):
    # a graph of G steps forks onto the streams and joins back.
    G = max(S, min(steps, max(100, prob.copies)) // S * S)  # every rotating copy, where steps allow
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    cap.wait_stream(main)
    with torch.cuda.graph(graph, stream=cap):
        for st in streams:
            st.wait_stream(cap)
        for i in range(G):
            one(i)
        for st in streams:
            cap.wait_stream(st)
    main.wait_stream(cap)
    graph.replay()  # untimed warm replay
    torch.cuda.synchronize(device)
    full, rest = divmod(steps, G)
    tail = None
    if rest:
        # the last `rest` steps as a graph of their own, so every timed step
        # is a replayed step whatever the step count
        tail = torch.cuda.CUDAGraph()
        cap.wait_stream(main)
        with torch.cuda.graph(tail, stream=cap):
            for st in streams:
                st.wait_stream(cap)
            for i in range(rest):
                one(i)
            for st in streams:
                cap.wait_stream(st)
        main.wait_stream(cap)
        tail.replay()  # untimed warm replay
        torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # as in time_device: the graphs are submitted while the device spins,
    # so the host's submission latency is not part of the measured time (a
    # serving loop submits its next graph while the previous one runs)
    torch.cuda._sleep(HOST_COVER_CYCLES)
    e0.record(main)
    for _ in range(full):
        graph.replay()
    if tail is not None:
        tail.replay()
    e1.record(main)
    torch.cuda.synchronize(device)
    h2d = ha.numel() * ha.element_size() + (hsa.numel() * hsa.element_size() if hsa is not None else 0)
    d2h = hc[0].numel() * hc[0].element_size()
    if record is not None:
        record["C"], record["host_C"] = C, hc
    return e0.elapsed_time(e1) / 1e3, h2d, d2h


def roofline(prob: Problem, sec_per_step: float, peaks: dict, peak_kind: str, traffic=None):
    if bound_of(prob.dtype, prob.M) == "hbm":
        achieved = prob.bytes / sec_per_step / 1e9
        peak = float(peaks["hbm_gbs"])
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"hbm_gbs ({peak_kind})",
                "algorithmic_bytes_per_launch": prob.bytes}
    ratio = DTYPE_RATIO[prob.dtype]
    base = float(peaks["bf16_tflops"])
    peak = base * ratio
    achieved = prob.flops / sec_per_step / 1e12
    out = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
           "frac": round(achieved / peak, 4), "traffic": traffic,
           "peak_source": f"bf16_tflops burst ({peak_kind}) x {ratio:g} nominal {prob.dtype}/bf16 ratio",
           "algorithmic_flops_per_launch": prob.flops}
    if peaks.get("bf16_tflops_sustained"):
        # beside it, the power-capped rate of a seconds-long cuBLAS loop
        sus = float(peaks["bf16_tflops_sustained"]) * ratio
        out["peak_sustained"] = round(sus, 1)
        out["frac_of_sustained"] = round(achieved / sus, 4)
    kind = {"bf16": "bf16", "fp16": "fp16", "e4m3": "e4m3", "e2m1": "e2m1"}.get(prob.dtype)
    if MMA_RATES is not None and kind in MMA_RATES["ratio_to_bf16"]:
        # the same measured bf16 peak times this GPU's measured MMA ratio for
        # the dtype, in place of the nominal ratio
        mr = MMA_RATES["ratio_to_bf16"][kind]
        out["measured_mma_ratio"] = mr
        out["peak_measured_ratio"] = round(base * mr, 1)
        out["frac_of_measured_ratio_peak"] = round(achieved / (base * mr), 4)
        if peaks.get("bf16_tflops_sustained"):
            out["frac_of_measured_ratio_sustained"] = round(
                achieved / (float(peaks["bf16_tflops_sustained"]) * mr), 4)
    # the other roofline too: the algorithmic bytes against the measured HBM
    # bandwidth, and the attainable rate min(peak, AI x bandwidth)
    hbm = float(peaks["hbm_gbs"])
    gbs = prob.bytes / sec_per_step / 1e9
    attainable = min(peak, prob.flops / prob.bytes * hbm / 1e3)
    out["hbm_GB/s"] = round(gbs, 1)
    out["frac_of_hbm"] = round(gbs / hbm, 4)
    out["attainable"] = round(attainable, 1)
    out["frac_of_attainable"] = round(achieved / attainable, 4)
    return out


def traffic_from_profiles(name: str):
    """DRAM bytes per launch recorded from an ncu capture, if a summary for
    this workload is committed under profiles/ (key `traffic_bytes_per_launch`)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            return json.load(f).get(name)
    except (OSError, ValueError):
        return None


def cpu_baseline(name: str, budget_s: float = 12.0):
    """The oracle as it stands, on this host's cores, over a bounded sample
    of rows of the workload; value in the metric's unit (TFLOP/s)."""
    import oracle
    from dense_gemm_preshuffle_gb300 import inputs
    ops = inputs.workload_operands(name)
    cores = oracle.num_threads()
    rows = 1
    t = oracle.time_gemm(ops, np.arange(rows))
    while t < 1.0 and rows < ops.M:
        rows = min(ops.M, rows * 2)
        t = oracle.time_gemm(ops, np.arange(rows))
    reps, total = 1, t
    while total + t < budget_s and reps < 1000:
        total += oracle.time_gemm(ops, np.arange(rows))
        reps += 1
    flops = 2.0 * rows * ops.N * ops.K * reps
    return {"value": flops / total / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x C rows [0,{rows}) of {ops.M} ({rows * ops.N} outputs, K={ops.K}), "
                      f"{total:.1f} s wall"}


def run_ours(args):
    import torch
    world, rank, local, pg = dist_setup(args)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    peaks, peak_kind = load_peaks()
    global MMA_RATES
    if int(os.environ.get("RANK", "0")) == 0 and not args.no_others:
        MMA_RATES = tensor_rates()
    import dense_gemm_preshuffle_gb300 as gp
    gp.load_library()

    clocks = ClockSampler(local).start()
    prob = Problem(args.workload, device)
    t_start = time.perf_counter()
    sec = time_device(prob, args.steps, args.warmup, pg, device)
    t_end = time.perf_counter()
    sec = max_over_ranks(pg, sec, device)
    clock_summary = clocks.summary(t_start, t_end)
    e2e_steps = max(10, min(args.steps, 2000))
    if args.no_e2e:
        e2e_sec, h2d, d2h = float("nan"), 0, 0
    else:
        e2e_sec, h2d, d2h = time_e2e(prob, e2e_steps, args.warmup, device)
        e2e_sec = max_over_ranks(pg, e2e_sec, device)
    trials = time_trials(prob, args.warmup, device)
    clocks.stop()

    per = sec / args.steps
    value = whole_job_value(world, prob.flops, args.steps, sec)
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": prob.dtype,
        "data": "synthetic, seeded (workload recipe)",
        "config": workload_config(prob.name, prob.M, prob.N, prob.K),
        "setup": {"parallelism": f"replicas x{world}",
                  "l2": f"inputs larger than L2: {prob.copies} rotating packed-B/A copies "
                        f"({prob.copies * prob.packed_bytes / 1e6:.0f} MB)",
                  "timing": "CUDA-graph replay of back-to-back gemm_run_ex launches, CUDA events",
                  "flags": "GP_RUN_DEFAULT" if B_DEFAULT_FLAGS else "GP_RUN_B_CONSTANT (weights packed once)"},
        "gpu_launches": args.steps,
        "e2e": {"value": None if args.no_e2e else round(world * prob.flops * e2e_steps / e2e_sec / 1e12, 3),
                "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_sec / e2e_steps * 1e3, 5), "steps": e2e_steps,
                "streams": E2E_STREAMS, "timing": "CUDA-graph replay of H2D copy + gemm_run_ex + D2H copy per step",
                "kind": f"{E2E_STREAMS} concurrent independent requests (throughput, not single-call latency)"},
        "roofline": roofline(prob, per, peaks, peak_kind, traffic_from_profiles(prob.name)),
        "trials": trials,
        "clocks": clock_summary,
        "gpu": gpu_record(device),
        "pack_b": {"us": round(prob.pack_us, 2), "bytes": prob.packed_bytes,
                   "GB/s": round(2 * prob.packed_bytes / (prob.pack_us * 1e-6) / 1e9, 1)},
    }
    del prob
    torch.cuda.empty_cache()
    if not args.no_others:
        # the headline workload through plain gemm_run (no scheduling flag)
        try:
            pd = Problem(args.workload, device)
            pd.flags = gp.GP_RUN_DEFAULT
            sd = max_over_ranks(pg, time_device(pd, args.steps, args.warmup, pg, device), device)
            out["b_default"] = {"us_per_step": round(sd / args.steps * 1e6, 3),
                                "roofline": roofline(pd, sd / args.steps, peaks, peak_kind, None),
                                "steps": args.steps, "flags": "GP_RUN_DEFAULT (plain gemm_run)"}
            del pd
            torch.cuda.empty_cache()
        except Exception as e:
            out["b_default"] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
        # the headline workload with its activation L2-resident, as the
        # previous kernel's output would be; B still rotates past L2
        try:
            pa = Problem(args.workload, device)
            pa.A = [pa.A[0]] * len(pa.A)
            sa_ = max_over_ranks(pg, time_device(pa, args.steps, args.warmup, pg, device), device)
            out["a_l2_resident"] = {"us_per_step": round(sa_ / args.steps * 1e6, 3),
                                    "roofline": roofline(pa, sa_ / args.steps, peaks, peak_kind, None),
                                    "steps": args.steps,
                                    "inputs": "one A buffer for every step (L2-resident, as a previous "
                                              "kernel's output); B rotating past L2"}
            del pa
            torch.cuda.empty_cache()
        except Exception as e:
            out["a_l2_resident"] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
        others = {}
        from dense_gemm_preshuffle_gb300 import inputs
        for name in inputs.ALL_WORKLOADS:
            if name == args.workload:
                continue
            try:
                p2 = Problem(name, device)
                steps2 = max(20, min(args.steps, 400), p2.copies)  # every rotating copy at least once
                s2 = time_device(p2, steps2, args.warmup, pg, device)
                s2 = max_over_ranks(pg, s2, device)
                r = roofline(p2, s2 / steps2, peaks, peak_kind, traffic_from_profiles(name))
                others[name] = {"us_per_step": round(s2 / steps2 * 1e6, 3),
                                "TFLOP/s": round(p2.flops * steps2 / s2 / 1e12, 2),
                                "GB/s": round(p2.bytes * steps2 / s2 / 1e9, 1), "roofline": r,
                                "steps": steps2, "pack_b_us": round(p2.pack_us, 2),
                                "trials": time_trials(p2, args.warmup, device)}
                del p2
                torch.cuda.empty_cache()
            except Exception as e:  # a workload whose kernel is not built yet
                others[name] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
        out["others"] = others
        # weight streaming as a run of independent calls (GP_RUN_INDEPENDENT):
        # each call on its own weights and output, overlapping its neighbours
        ind = {}
        for name in inputs.ALL_WORKLOADS:
            if not name.startswith(("int8", "w4a8")):
                continue
            try:
                p4 = Problem(name, device)
                p4.flags = gp.GP_RUN_B_CONSTANT | gp.GP_RUN_INDEPENDENT
                steps4 = max(20, min(args.steps, 2000))
                s4 = max_over_ranks(pg, time_device(p4, steps4, args.warmup, pg, device), device)
                ind[name] = {"us_per_step": round(s4 / steps4 * 1e6, 3),
                             "GB/s": round(p4.bytes * steps4 / s4 / 1e9, 1),
                             "roofline": roofline(p4, s4 / steps4, peaks, peak_kind, None),
                             "steps": steps4, "flags": "GP_RUN_B_CONSTANT | GP_RUN_INDEPENDENT"}
                del p4
                torch.cuda.empty_cache()
            except Exception as e:
                ind[name] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
        out["independent_stream"] = ind
        # the fused bias + GELU epilogue on each float workload, against the plain product
        epi = {}
        for name in inputs.WORKLOADS:
            if name.startswith(("int8", "w4a8")):
                continue
            try:
                p3 = Problem(name, device)
                steps3 = max(20, min(args.steps, 400), p3.copies)
                s_plain = time_device(p3, steps3, args.warmup, pg, device)
                gen = torch.Generator().manual_seed(99)
                p3.epilogue = "bias_gelu"
                p3.bias = torch.randn(p3.N, generator=gen).to(device)
                s_epi = time_device(p3, steps3, args.warmup, pg, device)
                s_plain = max_over_ranks(pg, s_plain, device)
                s_epi = max_over_ranks(pg, s_epi, device)
                epi[name] = {"epilogue": "bias_gelu", "us_per_step": round(s_epi / steps3 * 1e6, 3),
                             "plain_us_per_step": round(s_plain / steps3 * 1e6, 3),
                             "TFLOP/s": round(p3.flops * steps3 / s_epi / 1e12, 2), "steps": steps3}
                del p3
                torch.cuda.empty_cache()
            except Exception as e:
                epi[name] = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
        out["epilogues"] = epi
        out["quantize"] = time_quantizers(args, pg, device, peaks, peak_kind)
        if MMA_RATES is not None:
            out["tensor_rates"] = MMA_RATES
    if rank == 0:
        if not args.no_cpu:
            out["cpu_baseline"] = cpu_baseline(args.workload)
            if not args.no_others:
                # the oracle on the other workloads too, a short bounded
                # sample each (rows of C), for its rate per workload
                from dense_gemm_preshuffle_gb300 import inputs
                out["cpu_oracle_others"] = {name: cpu_baseline(name, budget_s=1.5)
                                            for name in inputs.ALL_WORKLOADS if name != args.workload}
        print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def run_reference(args):
    """The oracle on this host's cores: each step is a bounded sample (a set
    of C rows) of the same workload; rank 0 alone runs it."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from dense_gemm_preshuffle_gb300 import inputs
    ops = inputs.workload_operands(args.workload)
    cores = oracle.num_threads()
    # size each step so that warm-up + K steps take about a minute in total
    target = min(0.5, 60.0 / (args.steps + args.warmup))
    rows, cols = np.arange(1), None
    t_row = oracle.time_gemm(ops, rows)
    if t_row > target:
        ncols = max(1, int(ops.N * target / t_row))
        cols = np.arange(ncols)
    else:
        nrows = 1
        while nrows < ops.M and oracle.time_gemm(ops, np.arange(min(ops.M, nrows * 2))) < target:
            nrows = min(ops.M, nrows * 2)
        rows = np.arange(nrows)
    for _ in range(args.warmup):
        oracle.time_gemm(ops, rows, cols)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.time_gemm(ops, rows, cols)
    sec = time.perf_counter() - t0
    n_out = len(rows) * (ops.N if cols is None else len(cols))
    flops = 2.0 * n_out * ops.K * args.steps
    value = flops / sec / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": ops.dtype,
        "data": "synthetic, seeded (workload recipe)",
        "config": workload_config(args.workload, ops.M, ops.N, ops.K),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {n_out} of the {ops.M * ops.N} outputs of C "
                                   f"(rows [0,{len(rows)}), {'all' if cols is None else len(cols)} columns; K={ops.K})"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-others", action="store_true", help="skip the other workloads' lines")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline leg")
    ap.add_argument("--b-default", action="store_true",
                    help="call without GP_RUN_B_CONSTANT (B requested only after the previous kernel)")
    args = ap.parse_args()
    global B_DEFAULT_FLAGS
    B_DEFAULT_FLAGS = args.b_default
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
