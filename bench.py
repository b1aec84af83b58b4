#!/usr/bin/env python3
"""Benchmark of the pipelined, warp-specialized GEMM library on GB300.

One step = one f16 NT GEMM over the headline workload (default 8192^3 with
S = 4 ring slots, lhs [M,K] and rhs [N,K] f16 uniform in [-1,1] from seed 5,
fp32 accumulate, f16 out), launched through the C ABI.  The inputs stay resident in HBM during
the timed region and are larger than the 129 MB L2 (256 MB of operands), so
no L2 flush is needed between steps.

Prints ONE JSON line (rank 0):
  value / ms_per_step   -- device time of K back-to-back steps (CUDA events on
                           the launching stream, barrier + synchronize on both
                           sides, max over ranks)
  e2e                   -- the same metric through the C ABI with the inputs in
                           pinned HOST memory: each step copies lhs and rhs to
                           the device, runs the GEMM and copies out back
  roofline              -- the GEMM kernel's achieved TFLOP/s against the
                           measured dense 16-bit tensor peak
  cpu_baseline          -- the CPU oracle timed on a bounded sample of the
                           same workload on this host's cores, and whole on
                           each smaller workload (per_config; 1024^3 also on
                           one thread)
  clocks                -- nvidia-smi samples taken during the timed region
  configs               -- the other workloads (kernel-only timings): s32 NN
                           128x256x256, f16 NT 1024^3 S=2, 4096^3 S=4, the
                           ragged 4000x3000x2050 S=3 and the 8192^3 S=1..6 sweep
                           (each point after 0.25 s of warm-up, and the pipeline
                           cost model fitted to it), and 16 independent
                           1024^3 f16 / s32 GEMMs issued
                           on 1, 2, 4 or 8 streams (host concurrency)
                           and per-launch median / p10 / p90 at 4096^3, 8192^3

--impl reference times the CPU oracle instead (the slow reference arm).
With torchrun (N > 1) every rank runs an independent replica of the workload
(weak scaling; the GEMM has no exchange step).
"""
from __future__ import annotations

import argparse
import datetime
import functools
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

from pipelined_warp_specialized_gb300 import inputs  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "gemm_f16_nt_8192_traffic.txt")
KERNEL_SOURCES = [os.path.join(ROOT, "pipelined_warp_specialized_gb300", "csrc", f)
                  for f in ("gemm_f16_nt.cu", "ptx.cuh", "internal.h")]


# ---------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The maximum of x over all ranks (identity for one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_sha() -> str:
    """First 16 hex digits of sha256 over every source the f16 kernel compiles from."""
    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(M, N, K, S):
    """DRAM bytes per launch from the committed ncu summary of this shape and
    stage count, or None if absent, taken on another shape or S (S selects the
    tile) or on another version of the kernel."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    vals = {}
    with open(PROFILE_TRAFFIC) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    try:
        if vals.get("kernel_sha") != kernel_sha():
            return None
        if (int(vals["M"]), int(vals["N"]), int(vals["K"]), int(vals["stages"])) != (M, N, K, S):
            return None
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""
    # nvidia-smi's own sample time comes first: lines written to a pipe can
    # reach us in bursts, so their arrival time does not place them
    # (power.draw is a one-second average on this GPU generation, too slow for
    # a timed region of under a second; power.draw.instant is the sample)
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw.instant,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={self.interval}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)            # let the first sample land before timing starts

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        def sample_time(ln, arrived):
            try:        # local time, as time.time() sees it on the same machine
                return datetime.datetime.strptime(ln.split(",")[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return arrived
        rows = [ln for ts, ln in self.lines if t0 - 0.06 <= sample_time(ln, ts) <= t1 + 0.06] or \
            [ln for _, ln in self.lines[-3:]]
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in rows:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                sm.append(float(f[2]))
                smax.append(float(f[3]))
                power.append(float(f[4]))
            except ValueError:
                continue
            for name, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_median": statistics.median(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


class NvmlSampler:
    """SM clock, power and clock-event reasons read through NVML (the
    driver's management library, read-only queries) every `interval_ms`
    from a background thread, so that even a timed region of a few
    milliseconds holds samples; the same output as ClockSampler.  These are
    the values the driver reports, as nvidia-smi does: on GB300 they follow
    the load with a lag (the power reading is a window average), so within
    a region of tens of milliseconds they show at most the start of the
    power limit's effect."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch, device: int, interval_ms: float = 2.0):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        uuid = getattr(torch.cuda.get_device_properties(device), "uuid", None)
        ok = False
        if uuid is not None:
            ok = self.lib.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(), ctypes.byref(self.h)) == 0
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(device, ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.interval = interval_ms / 1e3
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None

    def _one(self):
        ct = self.ct
        mhz, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        t = time.time()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) != 0:       # NVML_CLOCK_SM
            return
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        self.reasons_fn(self.h, ct.byref(rs))
        self.samples.append((t, mhz.value, mw.value / 1e3, rs.value))

    def _run(self):
        while not self.stop_flag.is_set():
            self._one()
            time.sleep(self.interval)

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()
        time.sleep(0.05)

    def stop(self, t0, t1):
        self.stop_flag.set()
        self.thread.join(timeout=2)
        top = self.ct.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.ct.byref(top))
        self.lib.nvmlShutdown()
        rows = [x for x in self.samples if t0 <= x[0] <= t1]
        reasons = sorted({name for _, _, _, r in rows for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median([r[1] for r in rows]) if rows else None,
                "sm_mhz_min": min(r[1] for r in rows) if rows else None,
                "sm_max_mhz": top.value or None,
                "power_w_median": round(statistics.median([r[2] for r in rows]), 1) if rows else None,
                "reasons": reasons, "samples": len(rows),
                "source": f"NVML every {self.interval * 1e3:.0f} ms inside the timed region"}


# ---------------------------------------------------------------- our arm

def time_launches(fn, steps, warmup, torch, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_steady(fn, torch, stream, warm_s=0.25, timed_s=0.25):
    """Average ms per launch of fn() once the board has settled.

    The launch count is sized from a short probe so that every point of a
    sweep gets the same warm-up time and the same timed time: under the
    board's power limit the clock a launch sees depends on the load of the
    preceding fraction of a second, so equal launch COUNTS would hand later
    points the power state earlier ones left behind.
    """
    probe = time_launches(fn, 5, 3, torch, stream)
    warm = max(3, int(warm_s / (probe * 1e-3)))
    steps = max(5, int(timed_s / (probe * 1e-3)))
    return time_launches(fn, steps, warm, torch, stream)


def time_graph(fn, torch, per_graph=20, replays=20):
    """Average ms per launch of fn(stream), replayed from a CUDA graph.

    For launch-bound small problems: the graph removes the host-side cost of
    each call (Python, ctypes, argument checks), leaving the GPU time.
    """
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            fn(s)                       # first calls do the per-device set-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(per_graph):
            fn(s)
    g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(replays):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (replays * per_graph)


def e2e_pipelined(pws, torch, dev, a_h, b_h, c_h, stages, n_steps, warmup=2):
    """Average ms per step of host -> device -> GEMM -> host, pipelined over steps.

    Every step copies its lhs and rhs from pinned host memory, runs the GEMM
    through the C ABI and copies the result back to pinned host memory.  The
    three phases run on three streams with two device buffers per operand;
    events order each buffer's reuse (copy-in of step i+2 waits for the GEMM of
    step i; the GEMM of step i+2 waits for the copy-out of step i).
    """
    M, K = a_h.shape
    N = b_h.shape[0]
    s_in, s_mm, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    a = [torch.empty(M, K, dtype=torch.float16, device=dev) for _ in range(2)]
    b = [torch.empty(N, K, dtype=torch.float16, device=dev) for _ in range(2)]
    c = [torch.empty(M, N, dtype=torch.float16, device=dev) for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_mm = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def step(i):
        j = i % 2
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(ev_mm[j])          # the GEMM two steps back has read a[j], b[j]
            a[j].copy_(a_h, non_blocking=True)
            b[j].copy_(b_h, non_blocking=True)
            ev_in[j].record(s_in)
        s_mm.wait_event(ev_in[j])
        if used[j]:
            s_mm.wait_event(ev_out[j])             # the copy-out two steps back has read c[j]
        pws.gemm_f16_nt(a[j], b[j], c[j], stages=stages, stream=s_mm)
        ev_mm[j].record(s_mm)
        s_out.wait_event(ev_mm[j])
        with torch.cuda.stream(s_out):
            c_h.copy_(c[j], non_blocking=True)
            ev_out[j].record(s_out)
        used[j] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(n_steps):
        step(warmup + i)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n_steps


def per_launch_distribution(pws, torch, stream, shapes=((4096, 4), (8192, 4)), n=60, warmup=10):
    """Each of n back-to-back launches timed by its own pair of CUDA events on
    the launching stream (after `warmup` untimed ones): median, p10 and p90."""
    out = {}
    dev = torch.device("cuda")
    for M, S in shapes:
        a = torch.rand(M, M, device=dev, dtype=torch.float16) * 2 - 1
        b = torch.rand(M, M, device=dev, dtype=torch.float16) * 2 - 1
        c = torch.empty(M, M, device=dev, dtype=torch.float16)
        for _ in range(warmup):
            pws.gemm_f16_nt(a, b, c, stages=S, stream=stream)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        ev[0].record(stream)
        for i in range(n):
            pws.gemm_f16_nt(a, b, c, stages=S, stream=stream)
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        us = sorted(ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(n))
        pick = lambda q: us[min(n - 1, int(q * n))]
        out[f"f16_nt_{M}^3/S{S}/per_launch"] = {
            "median_us": round(pick(0.5), 1), "p10_us": round(pick(0.1), 1), "p90_us": round(pick(0.9), 1),
            "median_TFLOP_s": round(2 * M ** 3 / pick(0.5) / 1e6, 1),
            "median_frac_of_burst_peak": round(2 * M ** 3 / pick(0.5) / 1e6 / measured_peaks()[0]["bf16_tflops"], 4),
            "launches": n}
        del a, b, c
    return out


def concurrency_configs(pws, torch, G=16, stream_counts=(1, 2, 4, 8)):
    """Host concurrency: G independent GEMMs of one small shape, issued
    round-robin on n streams (fork from one stream, join back), captured in a
    CUDA graph so that the GPU, not the host's launch cost, decides how much
    of them overlaps.  Reported per batch of G."""
    out = {}
    dev = torch.device("cuda")
    wl = inputs.WORKLOADS["f16_nt_1024"]
    a, b = (torch.from_numpy(x).to(dev) for x in workload_inputs(wl.name))
    outs = [torch.empty(wl.M, wl.N, dtype=torch.float16, device=dev) for _ in range(G)]
    wl2 = inputs.WORKLOADS["s32_nn_128x256x256"]
    a2, b2 = torch.from_numpy(wl2.lhs()).to(dev), torch.from_numpy(wl2.rhs()).to(dev)
    outs2 = [torch.empty(wl2.M, wl2.N, dtype=torch.int32, device=dev) for _ in range(G)]
    cases = [(wl, "TFLOP_s", lambda i, st: pws.gemm_f16_nt(a, b, outs[i], stages=wl.stages[0], stream=st)),
             (wl2, "TOPS", lambda i, st: pws.gemm_s32_nn(a2, b2, outs2[i], stream=st))]
    for w, unit, call in cases:
        res = {}
        for ns in stream_counts:
            streams = [torch.cuda.Stream() for _ in range(ns)]

            def batch(s0, streams=streams, call=call):
                for st in streams:
                    st.wait_stream(s0)
                for i in range(G):
                    call(i, streams[i % len(streams)])
                for st in streams:
                    s0.wait_stream(st)

            ms = time_graph(batch, torch, per_graph=4, replays=20)
            res[f"streams{ns}"] = {"us_per_batch": round(ms * 1e3, 1), unit: round(G * w.flops / ms / 1e9, 2)}
        out[f"{w.name}/x{G}_concurrent"] = res
    return out


def sweep_model(res, plan, pairs, hi=4):
    """The pipeline cost model (TileLang tutorial ch.22, section 1.1) fitted
    to the sweep's S = 1 and S = hi points (one tile throughout), and its
    prediction for S = 2 .. hi-1 beside the measurement."""
    from pipelined_warp_specialized_gb300 import cost_model
    mids = tuple(range(2, hi))
    if not all(f"S{s}" in res and res[f"S{s}"]["tile"] == res["S1"]["tile"] for s in (1, hi) + mids):
        return None
    units = plan["tiles"]                       # tiles, one wave of `pairs` CTA pairs at a time
    blocks = -(-units // pairs) * plan["k_blocks"]     # the busiest pair's K blocks
    t1, th = res["S1"]["us"], res[f"S{hi}"]["us"]
    c, latency = cost_model.fit(blocks, t1, th)
    pred = cost_model.predict_sweep(blocks, t1, th, mids)
    return {"fit": f"c and L per K block from S = 1 (B (L + c)) and S = {hi} (B c), "
                   "B = the busiest CTA pair's blocks",
            "blocks": blocks, "c_us": round(c, 4), "L_us": round(latency, 4),
            "saturation_S": round(cost_model.saturation_stages(c, latency), 2),
            **{f"S{s}": {"predicted_us": round(pred[s], 1), "measured_us": res[f"S{s}"]["us"],
                         "measured_over_predicted": round(res[f"S{s}"]["us"] / pred[s], 3)} for s in mids}}


def peaks_library():
    """The measurement kernels (_build/libpwspeaks.so, built with the library)."""
    import ctypes
    from pipelined_warp_specialized_gb300 import build as libbuild
    lib = ctypes.CDLL(libbuild.PEAKS_PATH)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.pws_peaks_imad.argtypes = [i32, i32, i32, vp, vp]
    lib.pws_peaks_imad.restype = i32
    lib.pws_peaks_empty.argtypes = [i32, i32, vp]
    lib.pws_peaks_empty.restype = i32
    lib.pws_peaks_imad_chains.restype = i32
    lib.pws_peaks_mma.argtypes = [i32, i32, ctypes.c_uint64, vp, vp, vp]
    lib.pws_peaks_mma.restype = i32
    lib.pws_peaks_mma_step_flops.restype = ctypes.c_longlong
    return lib


def tensor_rate(torch, stream, steps=8192):
    """The tensor pipe's dense f16 -> fp32 rate per SM per clock, measured:
    one CTA per SM issues `steps` K steps of four tcgen05.mma (M = 128,
    N = 256, K = 16) back to back from shared memory, timed in SM cycles
    (clock64) from the first issue to the last MMA's completion; the median
    over the CTAs of the second of two launches."""
    lib = peaks_library()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out = torch.zeros(2 * sms, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        rc = lib.pws_peaks_mma(sms, steps, 2_000_000_000, out.data_ptr(), status.data_ptr(), stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"pws_peaks_mma failed ({rc})")
        torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("pws_peaks_mma: a bounded wait gave up")
    v = out.cpu().numpy().reshape(sms, 2).astype(np.float64)
    flops = steps * lib.pws_peaks_mma_step_flops()
    per_clk = np.median(flops / v[:, 0])
    ghz = np.median(v[:, 0] / v[:, 1])
    return {"flop_per_clk_per_sm": round(float(per_clk), 1), "sms": sms,
            "sm_ghz_during": round(float(ghz), 3),
            "how": f"{sms} CTAs x {steps} K steps of 4 tcgen05.mma.cta_group::1.kind::f16 "
                   "(128 x 256 x 16) from one shared-memory tile pair, SM cycles from the first issue "
                   "to the last completion, median over CTAs"}


def s32_roofline(torch, stream, us, ops, grid_blocks=128, threads=256):
    """The s32 path's two bounds, measured here: the CUDA-core peak of 32-bit
    multiply-adds (each counted as 2 ops, like 2MNK) from a kernel of
    independent mad.lo.u32 chains on every SM, and the launch floor, an
    empty kernel with the s32 page problem's grid (8 x 16 blocks of 256
    threads), launched the same way and replayed from a CUDA graph."""
    lib = peaks_library()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    blocks, thr, iters = sms * 8, 256, 4096
    call = lambda: lib.pws_peaks_imad(blocks, thr, iters, sink.data_ptr(), stream.cuda_stream)
    ms = time_launches(call, 20, 5, torch, stream)
    imads = blocks * thr * iters * lib.pws_peaks_imad_chains()
    peak_tops = 2 * imads / ms / 1e9
    floor_ms = time_graph(lambda st: lib.pws_peaks_empty(grid_blocks, threads, st.cuda_stream), torch)
    return {"imad_peak_TOPS": round(peak_tops, 2),
            "imad_peak_how": f"{blocks} blocks x {thr} threads x {iters} x {lib.pws_peaks_imad_chains()} "
                             f"independent mad.lo.u32, 2 ops each, {ms * 1e3:.0f} us",
            "frac_of_imad_peak": round(ops / (us * 1e-6) / 1e12 / peak_tops, 4),
            "launch_floor_us": round(floor_ms * 1e3, 2),
            "launch_floor_how": f"empty kernel, {grid_blocks} blocks x {threads} threads, programmatic "
                                "dependent launch, CUDA-graph replay",
            "over_launch_floor": round(us / (floor_ms * 1e3), 2)}


def extra_configs(pws, torch, stream):
    """Kernel-only timings of every workload (inputs resident).  f16 entries
    carry their fraction of the measured burst dense 16-bit peak; those timed
    for 0.25 s of back-to-back launches (at the power limit's steady state)
    also carry their fraction of the measured sustained peak, the matching
    denominator for a kernel timed inside a long run."""
    out = {}
    dev = torch.device("cuda")
    burst = measured_peaks()[0]["bf16_tflops"]
    sustained = measured_peaks()[0]["bf16_tflops_sustained"]

    def fractions(tflops, steady):
        f = {"frac_of_burst_peak": round(tflops / burst, 4)}
        if steady:
            f["frac_of_sustained_peak"] = round(tflops / sustained, 4)
        return f
    wl = inputs.WORKLOADS["s32_nn_128x256x256"]
    a, b = (torch.from_numpy(x).to(dev) for x in workload_inputs(wl.name))
    c = torch.empty(wl.M, wl.N, dtype=torch.int32, device=dev)
    ms_eager = time_launches(lambda: pws.gemm_s32_nn(a, b, c, stream=stream), 200, 20, torch, stream)
    ms = time_graph(lambda st: pws.gemm_s32_nn(a, b, c, stream=st), torch)
    out[wl.name] = {"us": round(ms * 1e3, 2), "TOPS": round(wl.flops / ms / 1e9, 3),
                    "GB_s": round((wl.M * wl.K + wl.K * wl.N + wl.M * wl.N) * 4 / ms / 1e6, 1),
                    "us_eager": round(ms_eager * 1e3, 2), "timing": "CUDA-graph replay (us), eager calls (us_eager)"}
    out[wl.name]["roofline"] = s32_roofline(torch, stream, ms * 1e3, wl.flops)
    ring = {}
    for s in range(2, 7):
        ms = time_graph(lambda st: pws.gemm_s32_nn_ring(a, b, c, stages=s, stream=st), torch)
        ring[f"S{s}"] = {"us": round(ms * 1e3, 2), "TOPS": round(wl.flops / ms / 1e9, 3)}
    out[wl.name + "/ring"] = ring
    for name in ("f16_nt_1024", "f16_nt_4096", "f16_nt_ragged_4000x3000x2050", "f16_nt_8192"):
        wl = inputs.WORKLOADS[name]
        a, b = (torch.from_numpy(x).to(dev) for x in workload_inputs(name))
        c = torch.empty(wl.M, wl.N, dtype=torch.float16, device=dev)
        # the ragged shape (rows no tensor map describes) is timed on each of
        # its paths: repacked into the library's fixed array + TMA (the
        # default: nothing allocated), read in place by the realigning
        # producer, repacked into pooled scratch + TMA (gemm_set_scratch_pool),
        # the no-alloc entry point (fixed array, rows 8-element aligned) and
        # the 4-byte cp.async producer
        variants = [("", 0, False, pws.gemm_f16_nt)]
        if name.startswith("f16_nt_ragged"):
            variants += [("in_place", pws.GEMM_DEBUG_IN_PLACE, False, pws.gemm_f16_nt),
                         ("pooled_repack", 0, True, pws.gemm_f16_nt),
                         ("noalloc", 0, False, pws.gemm_f16_nt_noalloc),
                         ("copy_producer", pws.GEMM_DEBUG_FORCE_COPY_PRODUCER, False, pws.gemm_f16_nt)]
        for suffix, flags, pool, call in variants:
            pws.gemm_set_debug_flags(flags)
            pws.gemm_set_scratch_pool(pool)
            try:
                plan = pws.gemm_f16_nt_plan(wl.M, wl.N, wl.K, a.data_ptr(), b.data_ptr(), c.data_ptr(), wl.stages[0])
                label = {0: "tma", 1: f"cp.async{plan['copy_bytes']}B",
                         2: "repack into pooled scratch+tma" if pool else "repack into the fixed array+tma",
                         3: "realign in place"}[plan["producer"]]
                res = {"producer": label, "cta_group": plan["cta_group"]}
                small = wl.flops < 2 ** 34        # launch-bound: time from a CUDA graph
                for s in wl.stages:
                    graph = small and plan["producer"] in (0, 3) and call is pws.gemm_f16_nt
                    if graph:
                        ms = time_graph(lambda st: call(a, b, c, stages=s, stream=st), torch)
                    else:
                        ms = time_steady(lambda: call(a, b, c, stages=s, stream=stream), torch, stream)
                    ps = pws.gemm_f16_nt_plan(wl.M, wl.N, wl.K, a.data_ptr(), b.data_ptr(), c.data_ptr(), s)
                    res[f"S{s}"] = {"us": round(ms * 1e3, 1), "TFLOP_s": round(wl.flops / ms / 1e9, 1),
                                    **fractions(wl.flops / ms / 1e9, not graph),
                                    "GB_s": round((wl.M * wl.K + wl.N * wl.K + wl.M * wl.N) * 2 / ms / 1e6, 1),
                                    "tile": f"{ps['bm']}x{ps['bn']}"}
                    res[f"S{s}"]["timing"] = ("CUDA-graph replay" if graph
                                              else "0.25 s warm-up, then 0.25 s of back-to-back launches")
            finally:
                pws.gemm_set_debug_flags(0)
                pws.gemm_set_scratch_pool(False)
            if name == "f16_nt_8192" and not suffix:
                pairs = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count // 2
                res["model"] = sweep_model(res, plan, pairs)
            out[name + ("/" + suffix if suffix else "")] = res
        if name == "f16_nt_8192":
            # the same sweep on one tile for every S (256 x 256 pairs; the
            # default switches to the 256 x 512 tile for S <= 4), so each step
            # of S changes the ring depth only, and the model fitted to S = 1
            # and S = 6 predicts S = 2 .. 5
            pws.gemm_set_debug_flags(pws.GEMM_DEBUG_FORCE_NARROW_TILE)
            try:
                res = {"producer": "tma", "cta_group": 2}
                for s in range(1, 7):
                    ms = time_steady(lambda: pws.gemm_f16_nt(a, b, c, stages=s, stream=stream), torch, stream)
                    res[f"S{s}"] = {"us": round(ms * 1e3, 1), "TFLOP_s": round(wl.flops / ms / 1e9, 1),
                                    **fractions(wl.flops / ms / 1e9, True),
                                    "tile": "256x256",
                                    "timing": "0.25 s warm-up, then 0.25 s of back-to-back launches"}
                plan_n = pws.gemm_f16_nt_plan(wl.M, wl.N, wl.K, a.data_ptr(), b.data_ptr(), c.data_ptr(), 6)
            finally:
                pws.gemm_set_debug_flags(0)
            pairs = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count // 2
            res["model"] = sweep_model(res, plan_n, pairs, hi=6)
            out[name + "/same_tile_256x256"] = res
        del a, b, c
    out.update(concurrency_configs(pws, torch))
    out.update(per_launch_distribution(pws, torch, stream))
    return out


def run_s32(args):
    """Times gemm_s32_nn alone on the s32 workload (back-to-back launches on
    one stream), e.g. to profile its kernel; the full bench reports it under
    `configs` with its roofline."""
    import torch
    import pipelined_warp_specialized_gb300 as pws
    pws.load_library()
    stream = torch.cuda.current_stream()
    wl = args.wl
    a, b = torch.from_numpy(wl.lhs()).cuda(), torch.from_numpy(wl.rhs()).cuda()
    c = torch.empty(wl.M, wl.N, dtype=torch.int32, device="cuda")
    ms = time_launches(lambda: pws.gemm_s32_nn(a, b, c, stream=stream), args.steps, args.warmup, torch, stream)
    if pws.gemm_device_status() != pws.GEMM_OK:
        raise RuntimeError("device status after timing")
    return {"metric": "s32 NN GEMM TOPS (eager launches)", "value": round(wl.flops / ms / 1e9, 3), "unit": "TOPS",
            "us_per_launch": round(ms * 1e3, 2), "steps": args.steps, "warmup": args.warmup,
            "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "K": wl.K}}


def run_ours(args, world, rank, local):
    import torch
    import pipelined_warp_specialized_gb300 as pws
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pws.load_library()
    stream = torch.cuda.current_stream(dev)
    M, N, K, S = args.M, args.N, args.K, args.stages
    flops = 2.0 * M * N * K
    # the seeded synthetic workload (distribution and seed: config.values)
    a_h = torch.from_numpy(args.wl.lhs()).pin_memory()
    b_h = torch.from_numpy(args.wl.rhs()).pin_memory()
    c_h = torch.empty(M, N, dtype=torch.float16).pin_memory()
    a = a_h.to(dev)
    b = b_h.to(dev)
    c = torch.empty(M, N, dtype=torch.float16, device=dev)

    def step():
        pws.gemm_f16_nt(a, b, c, stages=S, stream=stream)

    flags = pws.GEMM_DEBUG_FORCE_NARROW_TILE if args.tile == "narrow" else 0
    if args.in_place:
        flags |= pws.GEMM_DEBUG_IN_PLACE
    if flags:
        pws.gemm_set_debug_flags(flags)
    pws.gemm_set_scratch_pool(args.scratch_pool)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = pws.gemm_device_status()
    if status != pws.GEMM_OK:
        raise RuntimeError(f"device status after warm-up: {pws.gemm_status_string(status)}")

    sampler = None
    if not args.no_clocks:
        try:
            sampler = NvmlSampler(torch, local)
        except (OSError, AttributeError):
            sampler = ClockSampler(local)          # nvidia-smi, 50 ms apart
    if sampler:
        sampler.start()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    ms_total = e0.elapsed_time(e1)
    clocks = sampler.stop(t0, t1) if sampler else None
    ms_total = max_over_ranks(ms_total, world, dev)
    status = pws.gemm_device_status()
    if status != pws.GEMM_OK:
        raise RuntimeError(f"device status after timing: {pws.gemm_status_string(status)}")
    plan = pws.gemm_f16_nt_plan(M, N, K, a.data_ptr(), b.data_ptr(), c.data_ptr(), S)
    pws.gemm_set_debug_flags(0)
    pws.gemm_set_scratch_pool(False)
    ms = ms_total / args.steps
    value = world * flops / ms / 1e9          # TFLOP/s over all ranks

    # end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        n_e2e = max(3, min(args.steps, 30))
        ms_e2e = max_over_ranks(e2e_pipelined(pws, torch, dev, a_h, b_h, c_h, S, n_e2e), world, dev)
        e2e = {"value": round(world * flops / ms_e2e / 1e9, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int((M * K + N * K) * 2), "d2h_bytes_per_step": int(M * N * 2),
               "ms_per_step": round(ms_e2e, 4), "steps": n_e2e,
               "how": "pinned host lhs/rhs -> device, gemm_f16_nt, out -> pinned host, every step; "
                      "copy-in, GEMM and copy-out run on three streams with double-buffered device "
                      "operands, so step i's GEMM overlaps step i+1's copy-in and step i-1's copy-out"}

    peaks, peak_src = measured_peaks()
    long_region = ms_total > 1000.0
    peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    achieved = flops / ms / 1e9
    nw = plan["bn"] // (128 * plan["cta_group"])
    # producers 1 (copy) and 3 (realign in place) run the pair kernel's
    # multi-warp producer; 0 and 2 (repacked, then TMA) the TMA one
    pk = 1 if plan["cta_group"] == 2 and plan["producer"] in (1, 3) else 0
    launches_per_step = 2 if plan["producer"] == 2 else 1      # repack_rows_kernel, then the GEMM
    roofline = {"bound": "tensor",
                "kernel": f"gemm_f16_nt_kernel<{plan['cta_group']},{S},{nw},{pk},{plan['bk'] // 64}>",
                "tile": f"{plan['bm']}x{plan['bn']}",
                "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "peak_source": f"{peak_src} {'sustained' if long_region else 'burst'} dense bf16 "
                               "(f16 and bf16 share the tensor rate)",
                "traffic": profiled_traffic(M, N, K, S),
                "algorithmic_bytes_per_launch": int((M * K + N * K + M * N) * 2)}
    # the tensor pipe's own ceiling: SMs x the measured dense f16 flops per
    # SM per clock x a clock -- the SM's maximum, and the clock the
    # microbenchmark itself ran at (cycles over nanoseconds, in the kernel)
    # right after the timed region, with every tensor pipe busy: the power
    # limit lowers it.  The driver's clock readings are not used here: they
    # lag a load of milliseconds (2070 MHz and under 200 W read during a
    # region the microbenchmark then ran at 1.55 GHz)
    try:
        pipe = tensor_rate(torch, stream)
        at = pipe["sms"] * pipe["flop_per_clk_per_sm"] * pipe["sm_ghz_during"] * 1e9 / 1e12
        pipe.update({"ceiling_tflops_at_its_clock": round(at, 1),
                     "frac_of_ceiling_at_its_clock": round(achieved / at, 4)})
        if clocks and clocks.get("sm_max_mhz"):
            top = pipe["sms"] * pipe["flop_per_clk_per_sm"] * clocks["sm_max_mhz"] * 1e6 / 1e12
            pipe.update({"ceiling_tflops_at_max_clock": round(top, 1),
                         "frac_of_ceiling_at_max_clock": round(achieved / top, 4)})

    except (OSError, RuntimeError) as ex:
        pipe = {"unavailable": str(ex)}
    roofline["tensor_pipe"] = pipe

    extras = None
    if rank == 0 and world == 1 and not args.no_sweep and (M, N, K) == (8192, 8192, 8192) and args.tile == "auto":
        extras = extra_configs(pws, torch, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        del a, b, c
        cpu = cpu_baseline(M, N, K, args.cpu_seconds, a_h.numpy(), b_h.numpy())

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return None
    line = {
        "metric": f16_metric(M, N, K),
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": args.wl.name, "M": M, "N": N, "K": K, "stages": S,
                   "accumulate": "f32", "layout": "lhs[M,K] rhs[N,K] out[M,N] row-major",
                   "values": f"{args.wl.dist} (seed {args.wl.seed}) rounded to f16",
                   "parallelism": f"replicas x{world}",
                   "l2": ("inputs larger than L2 (no flush)" if (M * K + N * K) * 2 > L2_BYTES else
                          "inputs fit in L2 and are timed back to back without a flush (warm L2)")},
        "gpu_launches": args.steps * launches_per_step,
        "roofline": roofline, "e2e": e2e, "clocks": clocks, "cpu_baseline": cpu, "configs": extras,
    }
    return line


def f16_metric(M, N, K):
    """The metric's name for one f16 workload's shape."""
    size = f"{M}^3" if M == N == K else f"{M}x{N}x{K}"
    return f"f16 NT GEMM TFLOP/s at {size} (fraction of GB300 dense f16 tensor peak in roofline)"


# ---------------------------------------------------------------- CPU oracle

@functools.lru_cache(maxsize=None)
def workload_inputs(name):
    """The seeded operands of one of the smaller workloads, generated once per
    process (the configs' timings and the oracle's share them)."""
    wl = inputs.WORKLOADS[name]
    return wl.lhs(), wl.rhs()


def oracle_time(a, b, rows):
    """Times the oracle on the first `rows` rows of lhs against all of rhs."""
    import oracle
    t0 = time.perf_counter()
    oracle.gemm_f16_nt_f64(a[:rows], b)
    return time.perf_counter() - t0


def cpu_baseline(M, N, K, seconds, a, b):
    """The oracle as it stands on this host's cores, on a bounded sample of
    the workload (the first rows of the output, all columns, full K)."""
    import oracle
    threads = oracle.default_threads()
    probe_rows = max(1, threads)
    t = oracle_time(a, b, probe_rows)
    rows = int(max(1, min(M, probe_rows * max(1.0, seconds / max(t, 1e-3)))))
    t = oracle_time(a, b, rows)
    flops = 2.0 * rows * N * K
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {M} output rows x {N} columns, K={K} (f64 triple loop), {t:.1f} s",
            "per_config": oracle_per_config(threads)}


def oracle_per_config(threads):
    """The oracle on each smaller workload, whole (seconds and GFLOP/s, all
    host threads), and on the 1024^3 one with a single thread: about 6 s."""
    import oracle
    out = {}
    runs = [(name, threads) for name in ("s32_nn_128x256x256", "f16_nt_1024", "f16_nt_ragged_4000x3000x2050",
                                         "f16_nt_4096")]
    runs.append(("f16_nt_1024", 1))
    for name, nt in runs:
        wl = inputs.WORKLOADS[name]
        a, b = workload_inputs(name)
        fn = oracle.gemm_s32_nn if name.startswith("s32") else oracle.gemm_f16_nt_f64
        t0 = time.perf_counter()
        fn(a, b, nthreads=nt)
        dt = time.perf_counter() - t0
        key = name if nt == threads else f"{name}/1_thread"
        out[key] = {"s": round(dt, 4), "GFLOP_s": round(wl.flops / dt / 1e9, 2), "threads": nt}
    return out


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on this host's cores."""
    if rank != 0:
        return None
    import oracle
    M, N, K = args.M, args.N, args.K
    threads = oracle.default_threads()
    b = args.wl.rhs()
    a_probe = args.wl.lhs_rows(max(1, min(M, threads)))
    # size one step so the whole warm-up + timed run stays within ~90 s
    t = oracle_time(a_probe, b, max(1, threads))
    per_row = t / max(1, threads)
    budget = 90.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(M, budget / max(per_row, 1e-6))))
    a = args.wl.lhs_rows(rows)
    for _ in range(args.warmup):
        oracle.gemm_f16_nt_f64(a, b)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm_f16_nt_f64(a, b)
    dt = (time.perf_counter() - t0) / args.steps
    value = 2.0 * rows * N * K / dt / 1e12
    sample = f"{rows} of {M} output rows x {N} columns, K={K} per step (f64 triple loop)"
    return {
        "impl": "reference", "metric": f16_metric(M, N, K),
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.wl.name, "M": M, "N": N, "K": K, "stages": args.stages,
                   "accumulate": "f64 (the oracle)", "layout": "lhs[M,K] rhs[N,K] out[M,N] row-major",
                   "values": f"{args.wl.dist} (seed {args.wl.seed}) rounded to f16",
                   "parallelism": "host cores", "sample_rows": rows},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--stages", type=int, default=4,
                    help="ring slots S of the timed GEMM (4: the wide 256x512 pair tile, the fastest "
                         "sustained configuration on GB300; 5 and 6 run the 256x256 tile)")
    ap.add_argument("--workload", default="f16_nt_8192", choices=list(inputs.WORKLOADS),
                    help="the seeded workload of the timed GEMM (the s32 one times gemm_s32_nn alone, "
                         "for profiling)")
    ap.add_argument("--scratch-pool", action="store_true",
                    help="gemm_set_scratch_pool(1): operands TMA cannot address are repacked into pooled "
                         "scratch (by default: into the library's fixed array where they fit, else read "
                         "in place)")
    ap.add_argument("--in-place", action="store_true",
                    help="GEMM_DEBUG_IN_PLACE: operands TMA cannot address are read in place by the "
                         "realigning producer, never repacked")
    ap.add_argument("--tile", choices=["auto", "narrow"], default="auto",
                    help="narrow: the 256x256 pair tile for every S (GEMM_DEBUG_FORCE_NARROW_TILE), as in "
                         "the same-tile S sweep")
    ap.add_argument("--shape", default=None, help="M,N,K override (uniform [-1,1) inputs, seed 5)")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-workload timings")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.shape:
        M, N, K = (int(x) for x in args.shape.split(","))
        args.wl = inputs.Workload(f"f16_nt_{M}x{N}x{K}", "f16_nt", M, N, K, 5, "uniform", (args.stages,))
    else:
        args.wl = inputs.WORKLOADS[args.workload]
    args.M, args.N, args.K = args.wl.M, args.wl.N, args.wl.K
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    world, rank, local = dist_env()
    if args.wl.kind == "s32_nn":
        if args.impl == "reference" or world > 1:
            ap.error("the s32 workload is timed alone, on one GPU, for profiling")
        print(json.dumps(run_s32(args)), flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
