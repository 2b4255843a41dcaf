#!/usr/bin/env python3
"""Benchmark: effective causal attention TFLOP/s of the GB300 chunked-prefill GQA
attention (24 Q heads / 4 KV heads / head_dim 256, BF16, causal, scale 1/16).

One step = one call of gqa_prefill_attn over the whole workload (default: the
4096-token chunk at the end of a 32768-key prefix). Effective FLOPs count only
visible (query, key) pairs: 4 * head_dim * n_q_heads * pairs (2*d for QK^T and
2*d for PV per pair and head), masked and padded work excluded.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Timing: W untimed warm-up steps; then K steps, each timed with CUDA events on
the launching stream; L2 is flushed (a 256 MB buffer write, outside the events)
before every step; barrier + synchronize on both sides of the loop; the
per-rank sum is reduced with MAX over ranks. For N > 1 (torchrun, one process
per GPU) every rank runs an independent replica of the workload ("replicas
only": the path needs no exchange), and value = all ranks' FLOPs / max time.

--impl reference times the FP64 CPU oracle (the only other implementation)
on the host cores, on a bounded sample of rows of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from gqa_inputs import (SERVING_PAGE_SIZE, WORKLOADS, make_paged_cache, make_qkv,  # noqa: E402
                        make_varlen, make_workload, sample_rows)

METRIC = "effective causal attention TFLOPS and % of GB300 BF16 tensor peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "q4096_kv32768"
# The batched leg: a 4096-token chunked-prefill step shared by 8 requests, 512 new
# tokens each, over prefixes of 0, 4096, ..., 28672 keys.
VARLEN_BATCH = [(512, 512 + 4096 * i) for i in range(8)]
FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20   # GB300 L2 (rounded): decode inputs rotate over more than 4x this
D_ROTATE = 8           # at most this many decode K/V sets
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one attention-kernel
# launch from an ncu capture, keyed by workload, with the SHA-256 of the kernel
# source it was measured on; reported as null once the source no longer matches.
KNOWN_TRAFFIC: dict = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum (1 pass) on the full launch:
    # 807.79 MB read + 52.76 MB written.
    "q4096_kv32768": {"bytes": 860_547_072, "kernel_sha256": "d77efab2999d1c435473562ee86357e529220c117bf2ef17ed4e856fc2d48ad2"},
}


def visible_pairs(q_len: int, kv_len: int) -> int:
    p0 = kv_len - q_len
    return q_len * p0 + q_len * (q_len + 1) // 2


def effective_flops(w) -> int:
    return 4 * w.head_dim * w.n_q_heads * visible_pairs(w.q_len, w.kv_len)


def kernel_source_sha() -> str:
    path = os.path.join(ROOT, "gqa_chunked_prefill_gb300", "csrc", "attn_fwd_sm103.cu")
    return hashlib.sha256(open(path, "rb").read()).hexdigest()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def bf16_peak(peaks: dict, peak_kind: str):
    """BF16 tensor peaks: (burst, the roofline's denominator for a call timed alone;
    sustained, a seconds-long cuBLAS loop at the power cap, reported beside it as context
    when a long timed region meets the cap; source text)."""
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = peaks.get("bf16_tflops_sustained")
    return burst, (float(sustained) if sustained else None), \
        f"{peak_kind} bf16_tflops (burst; kernel timed alone)"


def sampled(fn, device_index: int):
    """Run fn() with the clock sampler around it; returns (fn's result, clock record)."""
    smp = clock_sampler(device_index)
    smp.start()
    smp.mark(True)
    try:
        out = fn()
    finally:
        smp.mark(False)
    return out, smp.stop()


# ----------------------------------------------------------------------------- clocks
class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (the driver's
    libnvidia-ml, called with ctypes) every ~2 ms in a thread, so that even a timed
    region of a few tens of milliseconds holds real samples. Read-only queries."""

    # nvmlClocksEventReason* bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.002):
        import ctypes
        self.period = period_s
        self.samples = []
        self.t_start = self.t_stop = None
        self.stop_flag = False
        self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        if self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle)) != 0:
            raise OSError("no NVML handle for " + uuid)
        get_reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.get_reasons = get_reasons or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)

    def _read(self):
        import ctypes
        mhz, mw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not self.stop_flag:
            ok = self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0
            self.nvml.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(mw))
            ok = ok and self.get_reasons(self.handle, ctypes.byref(rs)) == 0
            if ok:
                self.samples.append((time.time(), float(mhz.value), mw.value / 1000.0, rs.value))
            time.sleep(self.period)

    def start(self):
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.05)

    def mark(self, start: bool):
        if start:
            self.t_start = time.time()
        else:
            self.t_stop = time.time()

    def stop(self):
        self.stop_flag = True
        self.thread.join(timeout=2)
        window = [x for x in self.samples if self.t_start <= x[0] <= self.t_stop]
        reasons = sorted({name for x in window for bit, name in self.REASONS.items() if x[3] & bit})
        sm = [x[1] for x in window]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(sm),
                "power_w_max": max((x[2] for x in window), default=None),
                "source": "NVML every ~2 ms inside the timed region"}


def clock_sampler(device_index: int):
    """NVML sampler if the driver library answers, else nvidia-smi."""
    try:
        return NvmlClockSampler(device_index)
    except (OSError, AttributeError):
        return ClockSampler(device_index)


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.t_start = self.t_stop = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            gpu = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            gpu = str(device_index)
        self.cmd = ["nvidia-smi", "-i", gpu, f"--query-gpu={self.FIELDS}",
                    "--format=csv,noheader,nounits", "-lms", "100"]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()  # nvidia-smi takes a moment to print its first sample
        while not self.samples and time.time() - t0 < 5.0 and self.proc.poll() is None:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, start: bool):
        if start:
            self.t_start = time.time()
        else:
            self.t_stop = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        window = [s for t, s in self.samples if self.t_start and self.t_start <= t <= (self.t_stop or t)]
        note = None
        if not window:  # timed region shorter than the sampling period: nearest samples
            window = [s for _, s in self.samples[-3:]]
            note = "timed region shorter than the 100 ms sampling period; nearest samples"
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in window:
            parts = [x.strip() for x in s.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None,
               "reasons": sorted(reasons), "samples": len(sm)}
        if note:
            out["note"] = note
        return out


# ----------------------------------------------------------------------------- oracle
def oracle_sample(w, q, k, v, target_s: float, seed: int = 17):
    """Time the FP64 oracle on a row sample sized for ~target_s seconds.
    Returns (tflops, cores, description, rows, seconds)."""
    import oracle
    q64, k64, v64 = (t.double().numpy() for t in (q, k, v))
    cores = oracle.host_threads()
    p0 = w.kv_len - w.q_len
    calib = sample_rows(w.q_len, w.n_q_heads, 2 * cores, seed=seed + 1)
    t0 = time.perf_counter()
    oracle.attention(q64, k64, v64, w.scale, rows=calib, n_threads=cores)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(max(cores, min(w.q_len * w.n_q_heads, len(calib) * target_s / dt)))
    rows = sample_rows(w.q_len, w.n_q_heads, n, seed=seed)
    t0 = time.perf_counter()
    oracle.attention(q64, k64, v64, w.scale, rows=rows, n_threads=cores)
    secs = time.perf_counter() - t0
    toks = rows.numpy() // w.n_q_heads
    flops = float(np.sum(4.0 * w.head_dim * (p0 + toks + 1)))
    desc = (f"{len(rows)} of {w.q_len * w.n_q_heads} (token, head) rows of {w.name} "
            f"(stratified: first/middle/last tokens, all heads, seeded random rows), "
            f"{flops / 1e9:.1f} GFLOP of effective work in {secs:.2f} s")
    return flops / secs / 1e12, cores, desc, len(rows), secs


# ----------------------------------------------------------------------------- ranks
def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the architecture)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """MAX of a per-rank number over all ranks (identity when not distributed)."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_replica: int, max_ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every replica's work over the slowest rank's time."""
    return world * flops_per_replica / (max_ms_per_step * 1e-3) / 1e12


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--page-size", type=int, default=SERVING_PAGE_SIZE,
                    help="also time the paged-K/V entry point with this page size (0: skip)")
    ap.add_argument("--no-fp8", action="store_true", help="skip the quantised-QK^T leg")
    ap.add_argument("--no-varlen", action="store_true", help="skip the batched (varlen) leg")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode leg")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = WORKLOADS[args.workload]
    flops = effective_flops(w)

    if args.impl == "reference":
        return run_reference(args, w, flops, world, rank)

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    import gqa_chunked_prefill_gb300 as gqa

    q_cpu, k_cpu, v_cpu = make_workload(w)
    q, k, v = (t.to(dev) for t in (q_cpu, k_cpu, v_cpu))
    out = torch.empty_like(q)
    lse = torch.empty((w.q_len, w.n_q_heads), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(events=None):
        _, plan = gqa.gqa_prefill_attn_ex(q, k, v, out, lse, w.q_len, w.kv_len, w.n_q_heads,
                                          w.n_kv_heads, w.head_dim, w.scale, stream=stream,
                                          fwd_events=events)
        return plan

    for _ in range(args.warmup):
        flush.zero_()
        plan = call()
    torch.cuda.synchronize(dev)
    if gqa.gqa_prefill_poll(stream) != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for e in ev:  # torch creates the CUDA event on first record; the library records f0/f1 itself
        for x in e:
            x.record(stream)
    torch.cuda.synchronize(dev)
    sampler = clock_sampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark(True)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        s0, s1, f0, f1 = ev[i]
        s0.record(stream)
        call((f0, f1))
        s1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if sampler:
        sampler.mark(False)
    if pg:
        pg.barrier()
    step_ms = [a.elapsed_time(b) for a, b, _, _ in ev]
    fwd_ms = [a.elapsed_time(b) for _, _, a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), pg, dev)
    if gqa.gqa_prefill_poll(stream) != 0:
        raise RuntimeError("device-side wait timed out during the timed steps")
    clocks = sampler.stop() if sampler else None

    # ---- every workload shape, timed like the headline (same steps, flush, events) ----
    peaks_, peak_kind_ = load_peaks()

    def time_workload(wl):
        wq, wk, wv = (t.to(dev) for t in make_workload(wl))
        wo = torch.empty_like(wq)
        wlse = torch.empty((wl.q_len, wl.n_q_heads), dtype=torch.float32, device=dev)

        def wcall(events=None):
            return gqa.gqa_prefill_attn_ex(wq, wk, wv, wo, wlse, wl.q_len, wl.kv_len,
                                           wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.scale,
                                           stream=stream, fwd_events=events)[1]

        for _ in range(args.warmup):
            flush.zero_()
            wplan = wcall()
        wev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4))
               for _ in range(args.steps)]
        for e in wev:
            for x in e:
                x.record(stream)
        torch.cuda.synchronize(dev)

        def steps():
            for i in range(args.steps):
                flush.zero_()
                a, b, f0, f1 = wev[i]
                a.record(stream)
                wcall((f0, f1))
                b.record(stream)
            torch.cuda.synchronize(dev)

        _, wclocks = sampled(steps, local_rank)
        if gqa.gqa_prefill_poll(stream) != 0:
            raise RuntimeError(f"device-side error during {wl.name}")
        return ([a.elapsed_time(b) for a, b, _, _ in wev],
                [a.elapsed_time(b) for _, _, a, b in wev], wplan, wclocks)

    def workload_entry(wl, s_ms, f_ms, wplan, wclocks):
        wflops = effective_flops(wl)
        ms = max_over_ranks(sum(s_ms) / len(s_ms), pg, dev)
        kms = sum(f_ms) / len(f_ms)
        wpeak, wsust, _ = bf16_peak(peaks_, peak_kind_)
        return {"value": round(job_throughput(world, wflops, ms), 2), "unit": UNIT,
                "ms_per_step": round(ms, 4), "ms_median": round(statistics.median(s_ms), 4),
                "kernel_ms": round(kms, 4),
                "pct_of_peak": round(100.0 * wflops / (ms * 1e-3) / 1e12 / wpeak, 2),
                "roofline_frac": round(wflops / (kms * 1e-3) / 1e12 / wpeak, 4),
                "roofline_frac_vs_sustained":
                    round(wflops / (kms * 1e-3) / 1e12 / wsust, 4) if wsust else None,
                "clocks": {k_: wclocks.get(k_) for k_ in ("sm_mhz", "reasons")} if wclocks else None,
                "effective_gflop_per_step": round(wflops / 1e9, 2),
                "plan": {k_: wplan[k_] for k_ in ("variant", "head_rounds", "tail_items",
                                                  "tail_splits", "grid", "kernels_per_call")}}

    workloads = {}
    for name_, wl in WORKLOADS.items():
        if name_ == w.name:
            workloads[name_] = workload_entry(w, step_ms, fwd_ms, plan, clocks)
        else:
            workloads[name_] = workload_entry(wl, *time_workload(wl))
    torch.cuda.empty_cache()

    # ---- the same call with L2 left warm between steps (no flush) ---------------------
    warm_n = min(args.steps, 50)
    w_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(warm_n)]
    for a, b in w_ev:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize(dev)
    warm_ms = statistics.median(a.elapsed_time(b) for a, b in w_ev)

    # ---- end to end through the public call with host buffers ----------------------
    # Every step uploads its Q, K, V from pinned host memory, runs the call and
    # downloads out and LSE. Steps alternate between two device buffer sets, with
    # uploads and downloads on their own streams, so that step i+1's uploads and
    # step i-1's downloads overlap step i's attention, as a serving loop would
    # issue them; every step still moves all its bytes inside the timed region.
    e2e_steps = min(args.steps, 20)
    pin = lambda t: t.pin_memory()
    hq, hk, hv = pin(q_cpu), pin(k_cpu), pin(v_cpu)
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = (hq.numel() + hk.numel() + hv.numel()) * 2
    d2h = ho.numel() * 2 + hl.numel() * 4
    sets = [(q, k, v, out, lse),
            tuple(torch.empty_like(t) for t in (q, k, v, out, lse))]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(n):
        ev = lambda: torch.cuda.Event()
        uploaded, computed, downloaded = ([ev() for _ in range(n)] for _ in range(3))
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def upload(i):
            bq, bk, bv = sets[i % 2][:3]
            if i >= 2:
                h2d_s.wait_event(computed[i - 2])  # that set's Q/K/V are no longer read
            with torch.cuda.stream(h2d_s):
                bq.copy_(hq, non_blocking=True)
                bk.copy_(hk, non_blocking=True)
                bv.copy_(hv, non_blocking=True)
            uploaded[i].record(h2d_s)

        start.record(stream)
        h2d_s.wait_event(start)
        d2h_s.wait_event(start)
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            bq, bk, bv, bo, bl = sets[i % 2]
            stream.wait_event(uploaded[i])
            if i >= 2:
                stream.wait_event(downloaded[i - 2])  # that set's out/LSE were read back
            gqa.gqa_prefill_attn(bq, bk, bv, bo, bl, w.q_len, w.kv_len, w.n_q_heads,
                                 w.n_kv_heads, w.head_dim, w.scale, stream)
            computed[i].record(stream)
            d2h_s.wait_event(computed[i])
            with torch.cuda.stream(d2h_s):
                ho.copy_(bo, non_blocking=True)
                hl.copy_(bl, non_blocking=True)
            downloaded[i].record(d2h_s)
        stream.wait_event(downloaded[n - 1])
        end.record(stream)
        torch.cuda.synchronize(dev)
        return start.elapsed_time(end) / n

    e2e_run(2)
    e2e_ms = max_over_ranks(e2e_run(e2e_steps), pg, dev)

    # ---- the same workload with K/V read from a paged cache ------------------------
    paged = None
    if args.page_size > 0:
        kc_cpu, vc_cpu, table_cpu = make_paged_cache(k_cpu, v_cpu, args.page_size, seed=w.seed)
        kc, vc, table = kc_cpu.to(dev), vc_cpu.to(dev), table_cpu.to(dev)

        def pcall(events=None):
            return gqa.gqa_prefill_attn_paged_ex(
                q, kc, vc, table, kc.shape[0], args.page_size, out, lse, w.q_len, w.kv_len,
                w.n_q_heads, w.n_kv_heads, w.head_dim, w.scale, stream=stream,
                fwd_events=events)[1]

        for _ in range(3):
            flush.zero_()
            pcall()
        p_steps = min(args.steps, 100)
        pev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(p_steps)]
        for e in pev:
            for x in e:
                x.record(stream)
        torch.cuda.synchronize(dev)
        for i in range(p_steps):
            flush.zero_()
            s0, s1, f0, f1 = pev[i]
            s0.record(stream)
            pplan = pcall((f0, f1))
            s1.record(stream)
        torch.cuda.synchronize(dev)
        if gqa.gqa_prefill_poll(stream) != 0:
            raise RuntimeError("device-side error during the paged steps")
        p_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b, _, _ in pev) / p_steps, pg, dev)
        p_fwd = sum(a.elapsed_time(b) for _, _, a, b in pev) / p_steps
        paged = {"page_size": args.page_size, "num_pages": int(kc.shape[0]),
                 "block_table": "seeded permutation of the cache's pages; unused slots NaN",
                 "steps": p_steps, "value": round(job_throughput(world, flops, p_ms), 2),
                 "unit": UNIT, "ms_per_step": round(p_ms, 4), "kernel_ms": round(p_fwd, 4),
                 "kernels_per_call": pplan["kernels_per_call"]}
        del kc, vc, table

    # ---- the same workload with quantised QK^T (E4M3 codes + per-vector scales) ------
    fp8 = fp8pv = None
    if not args.no_fp8:
        stride = -(-w.kv_len // 4) * 4
        q8 = torch.empty(q.shape, dtype=torch.uint8, device=dev)
        qs = torch.empty((w.q_len, w.n_q_heads), dtype=torch.float32, device=dev)
        k8 = torch.empty(k.shape, dtype=torch.uint8, device=dev)
        ks = torch.empty((w.n_kv_heads, stride), dtype=torch.float32, device=dev)

        def quant_q():
            gqa.gqa_quantize_q_fp8(q, q8, qs, w.q_len, w.n_q_heads, w.head_dim, stream=stream)

        def quant_k():
            gqa.gqa_quantize_k_fp8(k, k8, ks, w.kv_len, w.n_kv_heads, w.head_dim, stride,
                                   stream=stream)

        def fcall(events=None):
            return gqa.gqa_prefill_attn_fp8qk_ex(
                q8, qs, k8, ks, stride, v, out, lse, w.q_len, w.kv_len, w.n_q_heads,
                w.n_kv_heads, w.head_dim, w.scale, stream=stream, fwd_events=events)[1]

        def timed(fn, n, with_fwd=False):
            evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(n)]
            for e in evs:
                for x in e:
                    x.record(stream)
            torch.cuda.synchronize(dev)
            for i in range(n):
                flush.zero_()
                evs[i][0].record(stream)
                fn((evs[i][2], evs[i][3])) if with_fwd else fn()
                evs[i][1].record(stream)
            torch.cuda.synchronize(dev)
            step = sum(a.elapsed_time(b) for a, b, _, _ in evs) / n
            fwd = sum(a.elapsed_time(b) for _, _, a, b in evs) / n if with_fwd else None
            return step, fwd

        quant_q()
        quant_k()
        for _ in range(3):
            flush.zero_()
            fplan = fcall()
        f_steps = min(args.steps, 100)
        (f_ms, f_fwd), f_clocks = sampled(lambda: timed(fcall, f_steps, with_fwd=True), local_rank)
        if gqa.gqa_prefill_poll(stream) != 0:
            raise RuntimeError("device-side error during the FP8 steps")
        f_ms = max_over_ranks(f_ms, pg, dev)
        # The quantisers are HBM-bound: timed on rotating copies of Q and K (each set of
        # copies over 4x L2, so every call reads cold input) with no flush, whose dirty
        # lines would share HBM with them.
        def rotating_us(make_call, nbytes):
            n_rot = max(2, min(D_ROTATE, -(-4 * L2_BYTES // nbytes) + 1))
            calls = [make_call(r) for r in range(n_rot)]
            for c in calls:
                c()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(40)]
            torch.cuda.synchronize(dev)
            # A call takes tens of microseconds, about what the host needs to issue one:
            # the host queues all of them while the GPU spins (~5 ms), so no event pair
            # holds GPU idle time waiting for the next launch.
            torch.cuda._sleep(10_000_000)
            for i, (a, b) in enumerate(ev):
                a.record(stream)
                calls[i % n_rot]()
                b.record(stream)
            torch.cuda.synchronize(dev)
            return sum(a.elapsed_time(b) for a, b in ev) / len(ev), n_rot

        def q_copy_call(r):
            src = q if r == 0 else q.clone()
            return lambda: gqa.gqa_quantize_q_fp8(src, q8, qs, w.q_len, w.n_q_heads, w.head_dim,
                                                  stream=stream)

        def k_copy_call(r):
            src = k if r == 0 else k.clone()
            return lambda: gqa.gqa_quantize_k_fp8(src, k8, ks, w.kv_len, w.n_kv_heads,
                                                  w.head_dim, stride, stream=stream)

        qq_ms, q_rot = rotating_us(q_copy_call, q.numel() * 2)
        qk_ms, k_rot = rotating_us(k_copy_call, k.numel() * 2)
        q_bytes = q.numel() * 3 + w.q_len * w.n_q_heads * 4   # BF16 in, E4M3 codes + scales out
        k_bytes = k.numel() * 3 + w.kv_len * w.n_kv_heads * 4
        # quantised PV as well: E4M3 V (per-channel scales, codes transposed) and E4M3 P
        vstride = -(-w.kv_len // 16) * 16
        v8 = torch.empty((w.n_kv_heads, w.head_dim, vstride), dtype=torch.uint8, device=dev)
        vs8 = torch.empty((w.n_kv_heads, w.head_dim), dtype=torch.float32, device=dev)
        gqa.gqa_quantize_v_fp8(v, v8, vs8, w.kv_len, w.n_kv_heads, w.head_dim, vstride,
                               stream=stream)

        def pvcall(events=None):
            return gqa.gqa_prefill_attn_fp8qkpv_ex(
                q8, qs, k8, ks, stride, v8, vs8, vstride, out, lse, w.q_len, w.kv_len,
                w.n_q_heads, w.n_kv_heads, w.head_dim, w.scale, stream=stream,
                fwd_events=events)[1]

        for _ in range(3):
            flush.zero_()
            pvplan = pvcall()
        (pv_ms, pv_fwd), pv_clocks = sampled(lambda: timed(pvcall, f_steps, with_fwd=True),
                                             local_rank)
        if gqa.gqa_prefill_poll(stream) != 0:
            raise RuntimeError("device-side error during the FP8 PV steps")
        pv_ms = max_over_ranks(pv_ms, pg, dev)
        qv_ms, v_rot = rotating_us(
            lambda r: (lambda src=(v if r == 0 else v.clone()): gqa.gqa_quantize_v_fp8(
                src, v8, vs8, w.kv_len, w.n_kv_heads, w.head_dim, vstride, stream=stream)),
            v.numel() * 2)
        fp8pv = {"steps": f_steps, "value": round(job_throughput(world, flops, pv_ms), 2),
                 "clocks": pv_clocks,
                 "unit": UNIT, "ms_per_step": round(pv_ms, 4), "kernel_ms": round(pv_fwd, 4),
                 "kernels_per_call": pvplan["kernels_per_call"],
                 "quantize_v_us": round(qv_ms * 1e3, 1),
                 "note": "QK^T and PV on E4M3 (kind::f8f6f4): Q, K per-vector scales, V "
                         "per-(KV head, channel) scales, P rounded to E4M3; V quantisation "
                         f"timed apart on {v_rot} rotating copies"}
        del v8
        fp8 = {"steps": f_steps, "value": round(job_throughput(world, flops, f_ms), 2),
               "clocks": f_clocks,
               "unit": UNIT, "ms_per_step": round(f_ms, 4), "kernel_ms": round(f_fwd, 4),
               "kernels_per_call": fplan["kernels_per_call"],
               "quantize_q_us": round(qq_ms * 1e3, 1), "quantize_k_us": round(qk_ms * 1e3, 1),
               "quantize_gbs": {"q": round(q_bytes / (qq_ms * 1e-3) / 1e9, 1),
                                "k": round(k_bytes / (qk_ms * 1e-3) / 1e9, 1),
                                "note": f"rotating {q_rot} Q / {k_rot} K copies, no flush"},
               "note": "QK^T on E4M3 codes (kind::f8f6f4), scales restored before the softmax; "
                       "PV in BF16. Step = the attention call; Q/K quantisation timed apart."}
        del q8, k8

    # ---- a batched step: the 4096-token chunk budget split over 8 requests ----------
    varlen = None
    if not args.no_varlen:
        lens = VARLEN_BATCH
        vq, vk, vv, cu_q, cu_k = make_varlen(lens, seed=w.seed + 7)
        vq, vk, vv = vq.to(dev), vk.to(dev), vv.to(dev)
        vout = torch.empty_like(vq)
        vlse = torch.empty((vq.shape[0], w.n_q_heads), dtype=torch.float32, device=dev)
        v_flops = sum(4 * w.head_dim * w.n_q_heads * (ql * (kl - ql) + ql * (ql + 1) // 2)
                      for ql, kl in lens)

        def vcall():
            gqa.gqa_prefill_attn_varlen(vq, vk, vv, vout, vlse, cu_q, cu_k, w.n_q_heads,
                                        w.n_kv_heads, w.head_dim, w.scale, stream=stream)

        def separate():
            for b in range(len(lens)):
                gqa.gqa_prefill_attn(vq[cu_q[b]:], vk[cu_k[b]:], vv[cu_k[b]:], vout[cu_q[b]:],
                                     vlse[cu_q[b]:], lens[b][0], lens[b][1], w.n_q_heads,
                                     w.n_kv_heads, w.head_dim, w.scale, stream)

        def timed_plain(fn, n):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)]
            for fn_ in (fn, fn, fn):
                flush.zero_()
                fn_()
            torch.cuda.synchronize(dev)
            for a, b in evs:
                flush.zero_()
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize(dev)
            return sum(a.elapsed_time(b) for a, b in evs) / n

        n_v = min(args.steps, 100)
        v_ms = max_over_ranks(timed_plain(vcall, n_v), pg, dev)
        s_ms = max_over_ranks(timed_plain(separate, n_v), pg, dev)
        if gqa.gqa_prefill_poll(stream) != 0:
            raise RuntimeError("device-side error during the varlen steps")
        varlen = {"batch": [list(x) for x in lens], "steps": n_v,
                  "effective_gflop_per_step": round(v_flops / 1e9, 2),
                  "value": round(job_throughput(world, v_flops, v_ms), 2), "unit": UNIT,
                  "ms_per_step": round(v_ms, 4), "separate_calls_ms": round(s_ms, 4),
                  "note": "one gqa_prefill_attn_varlen call vs one gqa_prefill_attn call per "
                          "sequence, same data"}
        del vq, vk, vv

    # ---- decode: one new token over the workload's prefix (HBM-bound) ------------------
    # Calls rotate over D_ROTATE distinct K/V sets (together more than 4x L2), so every call
    # reads K and V that no call touched in the last few hundred MB of traffic: cold reads
    # without a flush. (A flush by a 256 MB write leaves L2 full of dirty lines whose
    # write-back shares HBM with the K/V stream; that variant is reported alongside.)
    decode = None
    if not args.no_decode:
        d_len = 1
        kv_bytes = 2 * w.kv_len * w.n_kv_heads * w.head_dim * 2
        n_rot = max(2, min(D_ROTATE, -(-4 * L2_BYTES // kv_bytes) + 1))
        d_sets = [tuple(t.to(dev) for t in make_qkv(d_len, w.kv_len, w.seed + 11 + r))
                  for r in range(n_rot)]
        dout = torch.empty_like(d_sets[0][0])
        dlse = torch.empty((d_len, w.n_q_heads), dtype=torch.float32, device=dev)

        def dcall(i, st=None):
            dq, dk, dv = d_sets[i % n_rot]
            gqa.gqa_prefill_attn(dq, dk, dv, dout, dlse, d_len, w.kv_len, w.n_q_heads,
                                 w.n_kv_heads, w.head_dim, w.scale, st or stream)

        def timed(fn, n, flushed):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(n)]
            torch.cuda.synchronize(dev)
            for i, (a, b) in enumerate(ev):
                if flushed:
                    flush.zero_()
                a.record(stream)
                fn(i)
                b.record(stream)
            torch.cuda.synchronize(dev)
            return max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / n, pg, dev)

        for i in range(3 * n_rot):
            dcall(i)
        d_ms = timed(dcall, 50, False)
        df_ms = timed(lambda i: dcall(0), 20, True)
        # 50 calls between one event pair: consecutive calls overlap through programmatic
        # launch (an event recorded between two calls prevents that)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for i in range(50):
            dcall(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        db_ms = max_over_ranks(e0.elapsed_time(e1) / 50, pg, dev)
        # the same calls replayed from CUDA graphs, one per K/V set (how a serving loop
        # issues decode steps)
        side = torch.cuda.Stream(dev)  # graphs are captured off the default stream
        graphs = []
        for r in range(n_rot):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                dcall(r, side)
            graphs.append(g)
        torch.cuda.synchronize(dev)
        dg_ms = timed(lambda i: graphs[i % n_rot].replay(), 50, False)
        del graphs
        hbm = float(load_peaks()[0].get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        gbs = kv_bytes / (d_ms * 1e-3) / 1e9
        decode = {"q_len": d_len, "kv_len": w.kv_len, "steps": 50,
                  "us_per_call": round(d_ms * 1e3, 2),
                  "us_per_call_back_to_back": round(db_ms * 1e3, 2),
                  "us_per_graph_replay": round(dg_ms * 1e3, 2),
                  "us_per_call_write_flushed": round(df_ms * 1e3, 2), "unit": "GB/s",
                  "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
                               "unit": "GB/s", "frac": round(gbs / hbm, 4),
                               "algorithmic_bytes": kv_bytes},
                  "note": f"K + V read once per call (the bound); calls rotate over {n_rot} K/V "
                          "sets (inputs larger than 4x L2, no flush); us_per_call (events around "
                          "each call, the roofline's basis) and back-to-back (50 calls in one "
                          "event pair); the write-flushed variant re-reads one set after a 256 MB "
                          "L2 flush write"}
        del d_sets

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0

    peaks, peak_kind = load_peaks()
    ms_per_step = total_ms / args.steps
    value = job_throughput(world, flops, ms_per_step)
    fwd_avg_ms = sum(fwd_ms) / len(fwd_ms)
    achieved = flops / (fwd_avg_ms * 1e-3) / 1e12
    peak, peak_sust, peak_src = bf16_peak(peaks, peak_kind)
    mix = lambda pk: 1.0 / (0.5 / (2.0 * pk) + 0.5 / pk)
    if fp8:
        # QK^T (half the FLOPs) at the FP8 rate = measured BF16 x 2 (the nominal FP8:BF16
        # ratio), PV at the measured BF16 rate.
        f_ach = flops / (fp8["kernel_ms"] * 1e-3) / 1e12
        fp8["roofline"] = {"bound": "tensor", "achieved": round(f_ach, 2), "peak": round(mix(peak), 1),
                           "unit": "TFLOP/s", "frac": round(f_ach / mix(peak), 4),
                           "frac_vs_sustained":
                               round(f_ach / mix(peak_sust), 4) if peak_sust else None,
                           "peak_source": f"{peak_src}: QK^T at 2x, PV at 1x"}
    if fp8pv:
        # both halves at the FP8 rate: measured BF16 x 2 (the nominal FP8:BF16 ratio)
        pv_ach = flops / (fp8pv["kernel_ms"] * 1e-3) / 1e12
        fp8pv["roofline"] = {"bound": "tensor", "achieved": round(pv_ach, 2),
                             "peak": round(2.0 * peak, 1), "unit": "TFLOP/s",
                             "frac": round(pv_ach / (2.0 * peak), 4),
                             "frac_vs_sustained":
                                 round(pv_ach / (2.0 * peak_sust), 4) if peak_sust else None,
                             "peak_source": f"{peak_src} x 2 (QK^T and PV in E4M3)"}
    known = KNOWN_TRAFFIC.get(w.name)
    traffic = known["bytes"] if known and known["kernel_sha256"] == kernel_source_sha() else None

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "ms_median": round(statistics.median(step_ms), 4),
        "ms_min": round(min(step_ms), 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded BF16 N(0,1) Q/K/V of the workload's shape)",
        "config": {
            "workload": w.name, "q_len": w.q_len, "kv_len": w.kv_len, "n_q_heads": w.n_q_heads,
            "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "scale": w.scale, "causal": "bottom-right",
            "effective_gflop_per_step": round(flops / 1e9, 2),
            "l2": "flushed before every step (256 MB buffer write outside the step events)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "plan": {k_: plan[k_] for k_ in ("head_rounds", "tail_items", "tail_splits", "grid",
                                             "num_sms", "kernels_per_call")},
        },
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "roofline": {
            "bound": "tensor",
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_source": peak_src,
            "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "frac_vs_sustained": round(achieved / peak_sust, 4) if peak_sust else None,
            "traffic": traffic,
            "kernel": "gqa_attn_fwd_sm103_kernel",
            "kernel_ms": round(fwd_avg_ms, 4),
        },
        "warm_l2": {"value": round(job_throughput(world, flops, warm_ms), 2), "unit": UNIT,
                    "ms_median": round(warm_ms, 4), "steps": warm_n,
                    "note": "no L2 flush between steps (K/V of the previous step partly in L2)"},
        "e2e": {
            "value": round(job_throughput(world, flops, e2e_ms), 2),
            "unit": UNIT,
            "ms_per_step": round(e2e_ms, 4),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "steps": e2e_steps,
            "note": "uploads / call / downloads pipelined over two device buffer sets and three "
                    "streams; no L2 flush (each step's uploads stream 184 MB through L2)",
        },
        "workloads": workloads,
        "gpu_launches": args.steps * plan["kernels_per_call"],
        "paged": paged,
        "fp8qk": fp8,
        "fp8qkpv": fp8pv,
        "varlen": varlen,
        "decode": decode,
        "clocks": clocks,
        "wall_s_timed_loop": round(wall, 4),
    }
    if not args.no_cpu_baseline:
        tf, cores, desc, _, _ = oracle_sample(w, q_cpu, k_cpu, v_cpu, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(tf, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                                "cpu_model": cpu_model(), "sample": desc}
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def run_reference(args, w, flops, world, rank):
    """The FP64 oracle, as it stands, on the host cores (rank 0 only)."""
    if world > 1 and rank != 0:
        return 0
    q, k, v = make_workload(w)
    import oracle
    q64, k64, v64 = (t.double().numpy() for t in (q, k, v))
    cores = oracle.host_threads()
    p0 = w.kv_len - w.q_len
    per_step_s = max(0.05, min(6.0, 150.0 / (args.steps + args.warmup)))  # whole run ~150 s
    calib = sample_rows(w.q_len, w.n_q_heads, 2 * cores, seed=99)
    t0 = time.perf_counter()
    oracle.attention(q64, k64, v64, w.scale, rows=calib, n_threads=cores)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(max(cores, len(calib) * per_step_s / dt))
    total_s, total_flops = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        rows = sample_rows(w.q_len, w.n_q_heads, n, seed=1000 + i)
        t0 = time.perf_counter()
        oracle.attention(q64, k64, v64, w.scale, rows=rows, n_threads=cores)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            toks = rows.numpy() // w.n_q_heads
            total_flops += float(np.sum(4.0 * w.head_dim * (p0 + toks + 1)))
            total_s += dt
    value = total_flops / total_s / 1e12
    desc = (f"per step ~{n} of {w.q_len * w.n_q_heads} (token, head) rows of {w.name}, "
            f"stratified sample re-drawn each step; value = sampled effective FLOPs / oracle time")
    measured_ms = 1e3 * total_s / args.steps
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(measured_ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded BF16 N(0,1) Q/K/V of the workload's shape, widened to FP64)",
        "config": {"workload": w.name, "q_len": w.q_len, "kv_len": w.kv_len, "n_q_heads": w.n_q_heads,
                   "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "scale": w.scale,
                   "effective_gflop_per_step": round(flops / 1e9, 2),
                   "note": "each step computes a sample of the workload's rows; ms_per_step is "
                           "the measured oracle time of one sampled step"},
        "full_workload": {"ms_per_step": round(1e3 * flops / (value * 1e12), 3),
                          "extrapolated": True,
                          "note": "the whole workload at the sampled rate (not measured)"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
