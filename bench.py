"""Benchmark: overlap-save FIR output throughput (GS/s) on GB300, with its roofline fraction.

One step is one pass of the whole hot path -- the fused block kernel over one call's input
(steps 3-5 of the overlap-save claim in "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法",
zl.czvv.com/42398539.html, plus the state carry) -- for the chosen workload (default C5, the largest single-GPU
workload: complex64, k = 2048 blocks of L = 49152, N = 65536 with the response H given, one
call).  The C4 workload's step is its stream of 64 calls.  With the default workload the line
also carries, under "also", the same measurement of C3 (k = 1024 blocks of L = 24577,
N = 32768), the other long-transform workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C5] [--also C3,...]
                  [--blocks B] [--impl ours|reference]

`--blocks B` shortens a single-call workload to B blocks (for profiler captures of a smaller
case of the same kernel).  Prints one JSON line on rank 0.  Under torchrun rank g filters shard g of one stream of N
workload-sized shards on its own GPU, its state starting as the halo (the last M-1 samples of
shard g-1) -- weak scaling, no data-path collective -- and the time is the maximum over ranks.  `--impl reference` times the float64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "overlap-save FIR output GS/s on 1 GB300; % of HBM/FP32 roofline"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FP32_LANES_PER_SM = 128
PROFILE_DIR = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------------------- roofline arithmetic


def bytes_per_output(w: W.Workload) -> float:
    """Algorithmic HBM bytes per output sample: the gather reads N samples per L outputs
    (input plus the (M-1)/L overlap re-read) and the store writes one."""
    s = w.sample_bytes
    return s * (1.0 + (w.M - 1) / w.L) + s


def flops_per_output(w: W.Workload) -> float:
    """Nominal flops per output sample: 5 N log2 N per complex N-point FFT (radix-2 count),
    two transforms and a 6N-flop complex multiply per block of L outputs; a real block pair
    shares one complex transform."""
    per_block = 2 * 5 * w.N * math.log2(w.N) + 6 * w.N
    return per_block / w.L / (2 if w.real else 1)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", d
    return FALLBACK_HBM_GBS, "fallback", {}


def kernel_source_hash(files) -> str:
    """Hash of the named kernel sources (file names under the package's csrc/)."""
    csrc = os.path.join(ROOT, "frequency_domain_order_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(files):
        path = os.path.join(csrc, name)
        if not os.path.exists(path):
            return "missing:" + name
        with open(path, "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(config: str):
    """dram bytes per launch from a committed ncu summary for this workload, if it was taken
    on the current sources of that kernel (the files the summary lists); else None."""
    p = os.path.join(PROFILE_DIR, f"traffic_{config}.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != kernel_source_hash(d.get("source_files", [])):
        return None, d.get("source_hash")
    return float(d["dram_bytes_per_launch"]), d.get("source_hash")


# ----------------------------------------------------------------------------- clocks (NVML)

_NVML_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
                 0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
                 0x100: "display_clock_setting"}


class ClockSampler:
    """Reads SM and memory clocks and clock-event reasons through NVML (read-only queries)
    every `period` seconds on a background thread while the timed region runs."""

    def __init__(self, device_index: int, period: float = 0.002):
        self.ok = False
        self.samples = []
        self.mem_samples = []
        self.reasons = 0
        self.period = period
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            bus = self._bus_id(device_index)
            rc = -1
            if bus:
                rc = self.nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h))
            if rc != 0:
                rc = self.nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(self.h))
            if rc != 0:
                return
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = int(mx.value)
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 2, ctypes.byref(mx))  # 2: memory clock
            self.mem_max_mhz = int(mx.value)
            self.ok = True
        except OSError:
            return

    @staticmethod
    def _bus_id(idx):
        try:
            import torch
            pr = torch.cuda.get_device_properties(idx)
            return "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        except Exception:
            return None

    def _read(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk))
        mem = ctypes.c_uint()
        self.nv.nvmlDeviceGetClockInfo(self.h, 2, ctypes.byref(mem))
        self.mem_samples.append(int(mem.value))
        f = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        f(self.h, ctypes.byref(rs))
        return int(clk.value), int(rs.value)

    def __enter__(self):
        self._stop = threading.Event()
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def _run(self):
        while not self._stop.is_set():
            mhz, rs = self._read()
            self.samples.append(mhz)
            self.reasons |= rs
            time.sleep(self.period)

    def __exit__(self, *exc):
        self._stop.set()
        if self.ok:
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "mem_mhz": statistics.median(self.mem_samples) if self.mem_samples else None,
                "mem_max_mhz": self.mem_max_mhz,
                "samples": len(self.samples),
                "reasons": [n for b, n in _NVML_REASONS.items() if self.reasons & b and b != 0x1],
                "source": "NVML, sampled every 2 ms during the timed region"}


# ----------------------------------------------------------------------------- distributed


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- our arm


def buffer_sets(per_set_bytes: int) -> int:
    """How many input/output buffer sets the timed steps alternate between: at least two, and
    enough that together they exceed L2, so that no step finds its inputs left in L2 by an
    earlier one."""
    return max(2, min(1024, -(-int(1.25 * L2_BYTES) // max(1, int(per_set_bytes)))))


def l2_note(sets: int, footprint: int) -> str:
    return (f"inputs larger than L2: steps alternate between {sets} input/output buffer sets, "
            f"{footprint / 1e6:.0f} MB in total vs {L2_BYTES / 2**20:.0f} MiB L2")


def hold_stream(steps: int):
    """Occupy the stream with a clock-bounded sleep kernel (~1 ms plus ~30 us per step) while the
    host enqueues the timed steps, so that the host's submission time does not appear as idle
    time between steps on the device.  It runs before the first timing event."""
    import torch
    torch.cuda._sleep(int(2e6) + 60000 * steps)


NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s figure the filter's roofline is also quoted against

_FP32_PEAK = None


def measure_fp32_peak(stream) -> float:
    """FP32 TFLOP/s of the library's multiply-add probe (independent chains on every SM), the best
    of three launches timed with events on `stream`; measured once per process, outside the
    timed region."""
    global _FP32_PEAK
    if _FP32_PEAK is None:
        import torch
        from frequency_domain_order_gb300 import fir_os
        fir_os.fp32_probe(4096, stream)
        best = 0.0
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            flops = fir_os.fp32_probe(32768, stream)
            b.record(stream)
            b.synchronize()
            best = max(best, flops / (a.elapsed_time(b) * 1e-3) / 1e12)
        _FP32_PEAK = best
    return _FP32_PEAK


def fp32_block(achieved_tflops: float, peak_tflops: float, nominal_tflops: float, sms: int, sm_mhz: float,
               **extra):
    return dict(extra, achieved_tflops=achieved_tflops, peak_tflops=peak_tflops,
                peak_source="measured: fir_os_fp32_probe (independent multiply-add chains on every SM), "
                            "best of 3 launches, outside the timed region",
                nominal_peak_tflops=nominal_tflops,
                nominal_source=f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {sm_mhz:.0f} MHz (median sampled)",
                frac=achieved_tflops / peak_tflops)


def steps_per_graph(sets: int, launches_per_step: int, max_launches: int = 2048) -> int:
    """Consecutive steps captured in one CUDA graph: a multiple of the buffer sets (a replay ends
    on the set it began with), at least 8 steps, at most ~max_launches kernel launches."""
    r = sets * max(1, -(-8 // sets))
    while r > sets and r * launches_per_step > max_launches:
        r -= sets
    return r


def graph_replays(K: int, R: int):
    """(steps of each replay) covering exactly K steps: full replays of R, then the remainder."""
    full, rem = divmod(K, R)
    return [R] * full + ([rem] if rem else [])


def roofline_block(achieved_gbs, peak_gbs, peak_kind, traffic, bytes_launch, flops_launch, launch_ms,
                   fp32_peak, t_hbm, t_fp32):
    """The roofline of the dominant kernel against the slower of its two bounds: the bytes moved
    at the measured copy bandwidth, or the nominal flops at the measured FP32 peak (an FFT is
    plain FP32 arithmetic: "alu")."""
    common = {"traffic": traffic, "algorithmic_bytes_per_launch": bytes_launch,
              "algorithmic_flops_per_launch": flops_launch, "kernel_ms_per_launch": launch_ms,
              "t_hbm_us": t_hbm * 1e6, "t_fp32_us": t_fp32 * 1e6}
    if t_fp32 > t_hbm:
        achieved = flops_launch / (launch_ms * 1e-3) / 1e12
        return dict(common, bound="alu", achieved=achieved, peak=fp32_peak, unit="TFLOP/s",
                    frac=achieved / fp32_peak,
                    peak_source="measured FP32 peak (fir_os_fp32_probe, this run)",
                    hbm_achieved=achieved_gbs, hbm_frac=achieved_gbs / peak_gbs)
    return dict(common, bound="hbm", achieved=achieved_gbs, peak=peak_gbs, unit="GB/s",
                frac=achieved_gbs / peak_gbs,
                peak_source=(f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                             if peak_kind == "measured" else "fallback 6.8 TB/s"),
                nominal_peak=NOMINAL_HBM_GBS, frac_of_nominal=achieved_gbs / NOMINAL_HBM_GBS)


def step_stats(durations_ms):
    """(median, 20th percentile) of per-step device times in ms."""
    d = sorted(durations_ms)
    return statistics.median(d), d[min(len(d) - 1, int(0.2 * (len(d) - 1) + 0.5))]


def config_block(w: W.Workload, footprint: int, sets: int = 2):
    l2 = l2_note(sets, footprint) if footprint else "host CPU run (no GPU L2 involved)"
    return {
        "workload": f"{w.name}: {w.description}",
        "n_samples": w.n * w.channels, "channels": w.channels, "calls_per_step": len(w.calls),
        "M": w.M, "N": w.N, "L": w.L,
        "sample": "float32" if w.real else "complex64",
        "coefficients": "H given (complex64)" if w.coef == "freq" else "h taps",
        "l2": l2,
    }


def plan_time(fir_os, w: W.Workload, coef, kind, reps: int = 5):
    """Wall time of fir_os_plan_create (device allocations, step 1 -- the frequency response, or
    the scaling and reordering of a given H -- and the final synchronisation), median of `reps`
    plans created after the first."""
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        p = fir_os.Plan(w.M, w.N, coef, real=w.real, coef_kind=kind)
        times.append((time.perf_counter() - t0) * 1e3)
        p.close()
    return {"median": statistics.median(times), "min": min(times), "reps": reps,
            "what": ("fir_os_plan_create wall time: device allocations, step 1 "
                     + ("(scaling and reordering of the given H)" if kind == fir_os.COEF_FREQ else
                        "(float64 FFT of the taps on the device, rounded once)")
                     + ", synchronised; median of plans created after a first")}


def run_ours(args, w: W.Workload, world: int, rank: int, local: int, cpu_budget: float = None):
    import torch
    if cpu_budget is None:
        cpu_budget = args.cpu_budget

    from frequency_domain_order_gb300 import build as fbuild
    from frequency_domain_order_gb300 import fir_os

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl")
    if rank == 0 or not os.path.exists(fbuild.LIB):
        fbuild.build()
    barrier(world)

    if w.channels == 1:
        # rank g filters shard g of one stream of `world` workload-sized shards; its state
        # starts as the halo: the last M-1 samples of shard g-1 (zeros for shard 0)
        x = W.make_x_shard(w, rank)
        halo = (W.make_x_shard(w, rank - 1)[w.n - (w.M - 1):] if rank > 0
                else W.make_state0(w))
    else:
        # a bank of channels: rank g filters channels g C .. g C + C - 1 of a world-wide bank
        # (independent streams, each from a zero state)
        x = np.stack([W.make_x_shard(w, rank * w.channels + c) for c in range(w.channels)])
        halo = np.zeros((w.channels, w.M - 1), dtype=x.dtype)
    if w.coef == "freq":
        coef = torch.from_numpy(W.make_H_given(w)).to(dev)
        kind = fir_os.COEF_FREQ
    else:
        coef = torch.from_numpy(W.make_h_device(w)).to(dev)
        kind = fir_os.COEF_TIME
    plan = fir_os.Plan(w.M, w.N, coef, real=w.real, coef_kind=kind)
    plan_ms = plan_time(fir_os, w, coef, kind)
    if args.dft_engine == "tensor":
        plan.set_dft_engine(fir_os.DFT_TENSOR)
    sets = buffer_sets(2 * x.nbytes)
    xs = [torch.from_numpy(x).to(dev) for _ in range(sets)]
    ys = [torch.empty_like(xs[0]) for _ in range(sets)]
    sts = [torch.from_numpy(halo.copy()).to(dev) for _ in range(sets)]
    footprint = sets * 2 * x.nbytes
    stream = torch.cuda.current_stream(dev)

    def call(k, off, c, strm):
        if w.channels == 1:
            plan.execute(xs[k][off: off + c], ys[k][off: off + c], sts[k], strm)
        else:
            plan.execute_batched(xs[k][:, off: off + c], ys[k][:, off: off + c], sts[k], strm)

    def step(i, evs=None):
        k = i % sets
        off = 0
        for q, c in enumerate(w.calls):
            if evs is not None:
                evs[q][0].record(stream)
            call(k, off, c, stream)
            if evs is not None:
                evs[q][1].record(stream)
            off += c

    ncall = len(w.calls)
    K = args.steps
    graphs = None
    if not args.direct:
        # consecutive steps (cycling through the buffer sets) captured into CUDA graphs and
        # replayed: one graph launch per R steps instead of per step, and programmatic dependent
        # launch overlaps each call's set-up with the previous call's end across step boundaries
        # too.  Every step still runs every call of the workload.
        for k in range(sets):
            step(k)
        torch.cuda.synchronize()
        R = steps_per_graph(sets, ncall)

        def capture(nsteps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                cap = torch.cuda.current_stream(dev)
                for i in range(nsteps):
                    off = 0
                    for c in w.calls:
                        call(i % sets, off, c, cap)
                        off += c
            return g
        graphs = {n: capture(n) for n in set(graph_replays(K, R))}
        for _ in range(-(-args.warmup // max(graphs))):
            graphs[max(graphs)].replay()
    else:
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()
    plan.device_status()

    runs = graph_replays(K, R) if graphs is not None else [1] * K
    nev = 1 if graphs is not None else ncall
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(nev)] for _ in runs]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        hold_stream(len(runs))
        for i, n in enumerate(runs):
            if graphs is None:
                step(i, ev[i])
            else:
                ev[i][0][0].record(stream)
                graphs[n].replay()
                ev[i][0][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier(world)
    plan.device_status()
    total_ms = ev[0][0][0].elapsed_time(ev[-1][-1][1])
    # per launch of the block kernel (each call is one launch; the state is written in-kernel):
    # the timed device time over the launches it holds
    launch_ms = total_ms / (K * ncall)
    step_ms = [s_ev[0][0].elapsed_time(s_ev[-1][1]) / n for s_ev, n in zip(ev, runs)]
    ms_step = reduce_max(total_ms / K, world, dev)
    launches_per_step = sum(plan.launches(c) for c in w.calls)

    total = w.n * w.channels  # output samples of one step on one GPU
    value = world * total / (ms_step * 1e-3) / 1e9
    peak, peak_kind, peaks = measured_peaks()
    bytes_step = total * bytes_per_output(w)
    bytes_launch = bytes_step / ncall
    achieved = bytes_launch / (launch_ms * 1e-3) / 1e9
    traffic, _ = profiled_traffic(w.name)
    clk = clocks.summary()
    sm_mhz = clk["sm_mhz"] if clk else (peaks.get("sm_max_mhz") or 2070.0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fp32_nominal = sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    fp32_peak = measure_fp32_peak(stream)
    med_ms, p20_ms = step_stats(step_ms)
    flops_step = total * flops_per_output(w)
    t_hbm = bytes_step / (peak * 1e9)
    t_fp32 = flops_step / (fp32_peak * 1e12)

    # end to end through the host-buffer entry point (pinned memory, copies in the timed region)
    # (a bank of channels: one host-buffer call per channel)
    xh = torch.from_numpy(x).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    sh = torch.zeros((w.channels, w.M - 1) if w.channels > 1 else (w.M - 1,), dtype=xh.dtype).pin_memory()

    def e2e_step():
        for ch in range(w.channels):
            xr, yr, sr = (xh[ch], yh[ch], sh[ch]) if w.channels > 1 else (xh, yh, sh)
            off = 0
            for c in w.calls:
                plan.execute_host(xr[off: off + c], yr[off: off + c], sr, stream)
                off += c

    for _ in range(max(1, min(args.warmup, 3))):
        e2e_step()
    e2e_steps = max(1, min(K, args.e2e_steps))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = reduce_max((time.perf_counter() - t0) / e2e_steps, world, dev)
    sb = w.sample_bytes
    e2e = {"value": world * total / e2e_s / 1e9, "unit": "GS/s",
           "h2d_bytes_per_step": w.channels * (w.n * sb + len(w.calls) * (w.M - 1) * sb),
           "d2h_bytes_per_step": w.channels * (w.n * sb + len(w.calls) * (w.M - 1) * sb),
           "steps": e2e_steps,
           "path": "fir_os_execute_host on page-locked host buffers: " + (
               "the fused kernel reads x and writes y and the state in host memory in place over "
               "the host link" if plan.kernel()["kind"] == "cta" else
               "chunks of ~2^21 samples copied in and out by the copy engines, pipelined against "
               "the kernel")}

    out = {
        "metric": METRIC, "value": value, "unit": "GS/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "ms_per_step_median": med_ms,
        "ms_per_step_p20": p20_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(config_block(w, footprint, sets),
                       parallelism=(f"{world} GPUs, each filtering one workload-sized shard of a "
                                    f"{world}-shard stream with the previous shard's last M-1 samples "
                                    f"as its state (no collective on the data path)")
                       if world > 1 else "1 GPU"),
        "roofline": roofline_block(achieved, peak, peak_kind, traffic, bytes_launch, flops_step / ncall, launch_ms,
                                   fp32_peak, t_hbm, t_fp32),
        "fp32": fp32_block(flops_step / ncall / (launch_ms * 1e-3) / 1e12, fp32_peak, fp32_nominal, sms, sm_mhz,
                           nominal_flops_per_output=flops_per_output(w)),
        "metric_roofline": {"t_hbm_us": t_hbm * 1e6, "t_fp32_us": t_fp32 * 1e6,
                            "bound": "hbm" if t_hbm >= t_fp32 else "fp32",
                            "frac": max(t_hbm, t_fp32) / (ms_step * 1e-3)},
        "e2e": e2e,
        "gpu_launches": K * launches_per_step,
        "launch_mode": (f"CUDA graphs of {max(runs)} consecutive steps (cycling through the buffer sets), "
                        f"replayed {len(runs)} times; per-step median and p20 are over replays"
                        if graphs is not None else "direct launches"),
        "clocks": clk,
        "kernel": dict(plan.kernel(), dft_engine=args.dft_engine),
        "plan_ms": plan_ms,
        "wall_s_timed_region": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # (a bank of channels: the oracle on channel 0, the same per-sample work)
        x0 = x if w.channels == 1 else x[0]
        out["cpu_baseline"] = cpu_baseline(w, x0, budget_s=cpu_budget)
        pc = single_thread_overlap_save(w, x0, budget_s=min(3.0, cpu_budget))
        pc["gpu_over_cpu"] = out["value"] / pc["value"]
        out["page_comparison"] = pc
    plan.close()
    return out


# ----------------------------------------------------------------------------- oracle legs


def _oracle_outputs(oracle, x, h, M: int, s: int, count: int):
    """The oracle's outputs s .. s + count of the stream x (S0 = 0): one call on the slice with
    the M-1 samples before it as its state, so that only the slice is marshalled."""
    hist = M - 1
    st = np.zeros(hist, dtype=x.dtype)
    lo = max(0, s - hist)
    if hist:
        st[hist - (s - lo):] = x[lo:s]
    return oracle.direct(x[s: s + count], h, st)[0]


def cpu_baseline(w: W.Workload, x, budget_s: float = 12.0):
    """Time the float64 oracle (direct convolution, all host cores) on a bounded sample of
    the workload: the first outputs of the stream, as many as fit the time budget."""
    import oracle
    h = W.oracle_h(w)
    probe = min(w.n, max(w.L, 1 << 16))
    t0 = time.perf_counter()
    _oracle_outputs(oracle, x, h, w.M, 0, probe)
    rate = probe / max(time.perf_counter() - t0, 1e-6)
    count = int(min(w.n, max(w.L, rate * budget_s)))
    t0 = time.perf_counter()
    _oracle_outputs(oracle, x, h, w.M, 0, count)
    dt = time.perf_counter() - t0
    return {"value": count / dt / 1e9, "unit": "GS/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"first {count} of {w.n} outputs ({count / w.n:.1%}), float64 direct "
                      f"convolution with M={w.M} taps, OpenMP over outputs"}


def single_thread_overlap_save(w: W.Workload, x, budget_s: float = 3.0):
    """The page's own comparison, as context: a single-thread CPU overlap-save (the oracle's own
    radix-2 FFT, float64, one core) over the first whole blocks of the workload, as many as fit
    the time budget."""
    import oracle
    h = W.oracle_h(w)
    H = oracle.freq_response(h, w.N)
    span = w.L
    blocks = 1
    t0 = time.perf_counter()
    oracle.overlap_save(x[: blocks * span], H, w.M)
    per_block = max(time.perf_counter() - t0, 1e-6)
    blocks = int(max(1, min(w.n // span, budget_s / per_block)))
    t0 = time.perf_counter()
    oracle.overlap_save(x[: blocks * span], H, w.M)
    dt = time.perf_counter() - t0
    return {"kind": "single-thread CPU overlap-save: the oracle's own radix-2 FFT in float64 on one core",
            "value": blocks * span / dt / 1e9, "unit": "GS/s", "cores": 1, "seconds": dt,
            "sample": f"first {blocks} blocks of {w.L} outputs ({blocks * span / w.n:.2%} of the stream)",
            "page_claim": "more than 100x over a single-thread CPU overlap-save (no hardware stated)"}


def run_reference(args, w: W.Workload, world: int, rank: int):
    """The oracle as the reference arm: each step evaluates a bounded contiguous sample of
    outputs; the whole run is sized to end within a few minutes."""
    if rank != 0:
        return None
    import oracle
    x = W.make_x(w)
    h = W.oracle_h(w)
    probe = min(w.n, 1 << 15)
    t0 = time.perf_counter()
    _oracle_outputs(oracle, x, h, w.M, 0, probe)
    rate = probe / max(time.perf_counter() - t0, 1e-6)
    per_step_s = min(0.5, 120.0 / max(1, args.steps + args.warmup))
    count = int(max(64, min(w.n, rate * per_step_s)))
    rng = np.random.Generator(np.random.PCG64(99))
    starts = rng.integers(0, max(1, w.n - count), args.steps + args.warmup)
    for i in range(args.warmup):
        _oracle_outputs(oracle, x, h, w.M, int(starts[i]), count)
    t0 = time.perf_counter()
    for i in range(args.steps):
        _oracle_outputs(oracle, x, h, w.M, int(starts[args.warmup + i]), count)
    dt = (time.perf_counter() - t0) / args.steps
    value = count / dt / 1e9
    sample = (f"{count} contiguous outputs per step at seeded random offsets "
              f"({count / w.n:.3%} of the {w.n}-sample stream), float64 direct convolution")
    return {
        "metric": METRIC, "value": value, "unit": "GS/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": config_block(w, 0),
        "cpu_baseline": {"value": value, "unit": "GS/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GS/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ----------------------------------------------------------------------------- channelizer

CHAN_METRIC = "polyphase channelizer input GS/s on 1 GB300; % of HBM roofline"


def chan_bytes_per_input(c) -> float:
    """Input read once, K complex64 outputs written per D inputs (prototype and state ignored)."""
    return c.sample_bytes + 8.0 * c.K / c.D


def chan_flops_per_input(c) -> float:
    """Nominal: the polyphase sums (2 Nh real, 4 Nh complex flops per output vector) and a
    K-point FFT (5 K log2 K) per output vector, per input sample."""
    return ((2 if c.real else 4) * c.Nh + 5.0 * c.K * math.log2(c.K)) / c.D


def run_chan(args, c, world: int, rank: int, local: int):
    import torch

    from frequency_domain_order_gb300 import build as fbuild
    from frequency_domain_order_gb300 import fir_os

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if rank == 0 or not os.path.exists(fbuild.LIB):
        fbuild.build()
    barrier(world)
    h = W.chan_prototype(c)
    x = W.chan_x(c)
    plan = fir_os.ChanPlan(c.K, c.D, torch.from_numpy(h.astype(np.float32)).to(dev), real=c.real)
    sets = buffer_sets(x.nbytes + c.nout * c.K * 8)
    xs = [torch.from_numpy(x).to(dev) for _ in range(sets)]
    ys = [torch.empty((c.nout, c.K), dtype=torch.complex64, device=dev) for _ in range(sets)]
    sts = [torch.zeros(c.Nh - 1, dtype=xs[0].dtype, device=dev) for _ in range(sets)]
    footprint = sets * (x.nbytes + c.nout * c.K * 8)
    stream = torch.cuda.current_stream(dev)
    for k in range(sets):
        plan.execute(xs[k], ys[k], sts[k], stream)
    torch.cuda.synchronize()
    # consecutive steps (cycling through the buffer sets) captured into CUDA graphs, as for the
    # filter: one graph launch per R steps
    K = args.steps
    R = steps_per_graph(sets, 2)

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(nsteps):
                plan.execute(xs[i % sets], ys[i % sets], sts[i % sets], torch.cuda.current_stream(dev))
        return g
    runs = graph_replays(K, R)
    graphs = {n: capture(n) for n in set(runs)}
    for _ in range(-(-args.warmup // max(graphs))):
        graphs[max(graphs)].replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in runs]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        hold_stream(len(runs))
        for (a, b), n in zip(ev, runs):
            a.record(stream)
            graphs[n].replay()
            b.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier(world)
    total_ms = ev[0][0].elapsed_time(ev[-1][1])
    launch_ms = total_ms / K  # per call (the filter-bank kernel and the state kernel)
    step_ms = [a.elapsed_time(b) / n for (a, b), n in zip(ev, runs)]
    ms_step = reduce_max(total_ms / K, world, dev)
    value = world * c.n / (ms_step * 1e-3) / 1e9
    peak, peak_kind, peaks = measured_peaks()
    bytes_step = c.n * chan_bytes_per_input(c)
    achieved = bytes_step / (launch_ms * 1e-3) / 1e9
    clk = clocks.summary()
    sm_mhz = clk["sm_mhz"] if clk else (peaks.get("sm_max_mhz") or 2070.0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fp32_nominal = sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    fp32_peak = measure_fp32_peak(stream)
    med_ms, p20_ms = step_stats(step_ms)
    flops_step = c.n * chan_flops_per_input(c)
    t_hbm = bytes_step / (peak * 1e9)
    t_fp32 = flops_step / (fp32_peak * 1e12)
    traffic, _ = profiled_traffic(c.name)

    # end to end: pinned input copied in, the call, the output copied back, every step
    xh = torch.from_numpy(x).pin_memory()
    yh = torch.empty((c.nout, c.K), dtype=torch.complex64).pin_memory()

    def e2e_step():
        xs[0].copy_(xh, non_blocking=True)
        plan.execute(xs[0], ys[0], sts[0], stream)
        yh.copy_(ys[0], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(1, min(K, args.e2e_steps))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = reduce_max((time.perf_counter() - t0) / e2e_steps, world, dev)
    out = {
        "metric": CHAN_METRIC, "value": value, "unit": "GS/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "ms_per_step_median": med_ms,
        "ms_per_step_p20": p20_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{c.name}: {c.description}", "n_samples": c.n, "K": c.K, "D": c.D,
                   "Nh": c.Nh, "sample": "float32" if c.real else "complex64",
                   "l2": l2_note(sets, footprint),
                   "parallelism": f"{world} GPUs, each its own copy of the stream" if world > 1 else "1 GPU"},
        "roofline": roofline_block(achieved, peak, peak_kind, traffic, bytes_step, flops_step, launch_ms,
                                   fp32_peak, t_hbm, t_fp32),
        "fp32": fp32_block(flops_step / (launch_ms * 1e-3) / 1e12, fp32_peak, fp32_nominal, sms, sm_mhz,
                           nominal_flops_per_input=chan_flops_per_input(c)),
        "metric_roofline": {"t_hbm_us": t_hbm * 1e6, "t_fp32_us": t_fp32 * 1e6,
                            "bound": "hbm" if t_hbm >= t_fp32 else "fp32",
                            "frac": max(t_hbm, t_fp32) / (ms_step * 1e-3)},
        "e2e": {"value": world * c.n / e2e_s / 1e9, "unit": "GS/s",
                "h2d_bytes_per_step": x.nbytes, "d2h_bytes_per_step": c.nout * c.K * 8, "steps": e2e_steps,
                "path": "pinned input copied in, fir_chan_execute, output copied back"},
        "gpu_launches": K * (2 if c.Nh > 1 else 1),
        "launch_mode": (f"CUDA graphs of {max(runs)} consecutive calls (cycling through the buffer sets), "
                        f"replayed {len(runs)} times; per-step median and p20 are over replays"),
        "clocks": clk,
        "wall_s_timed_region": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        h32 = h.astype(np.float32).astype(np.float64)
        probe = min(c.nout, 16)
        t0 = time.perf_counter()
        oracle.channelize_at(x, h32, c.K, c.D, None, np.arange(probe))
        rate = probe / max(time.perf_counter() - t0, 1e-6)
        rows = int(max(1, min(c.nout, rate * args.cpu_budget)))
        t0 = time.perf_counter()
        oracle.channelize_at(x, h32, c.K, c.D, None, np.arange(rows))
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": rows * c.D / dt / 1e9, "unit": "GS/s", "cores": oracle.num_threads(),
                               "kind": "oracle", "seconds": dt,
                               "sample": f"first {rows} of {c.nout} output vectors ({rows * c.D} input samples), "
                                         f"float64 defining sum, OpenMP over output vectors"}
    plan.close()
    return out


def run_chan_reference(args, c, world: int, rank: int):
    """The oracle as the reference arm on a channelizer workload: each step evaluates a bounded
    run of output vectors at a seeded offset."""
    if rank != 0:
        return None
    import oracle
    h = W.chan_prototype(c).astype(np.float32).astype(np.float64)
    x = W.chan_x(c)
    probe = min(c.nout, 16)
    t0 = time.perf_counter()
    oracle.channelize_at(x, h, c.K, c.D, None, np.arange(probe))
    rate = probe / max(time.perf_counter() - t0, 1e-6)
    per_step_s = min(0.5, 120.0 / max(1, args.steps + args.warmup))
    rows = int(max(1, min(c.nout, rate * per_step_s)))
    rng = np.random.Generator(np.random.PCG64(98))
    starts = rng.integers(0, max(1, c.nout - rows), args.steps + args.warmup)
    for i in range(args.warmup):
        oracle.channelize_at(x, h, c.K, c.D, None, np.arange(starts[i], starts[i] + rows))
    t0 = time.perf_counter()
    for i in range(args.steps):
        s0 = starts[args.warmup + i]
        oracle.channelize_at(x, h, c.K, c.D, None, np.arange(s0, s0 + rows))
    dt = (time.perf_counter() - t0) / args.steps
    value = rows * c.D / dt / 1e9
    sample = f"{rows} output vectors per step at seeded offsets ({rows * c.D} input samples), float64 defining sum"
    return {
        "metric": CHAN_METRIC, "value": value, "unit": "GS/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": f"{c.name}: {c.description}", "n_samples": c.n, "K": c.K, "D": c.D, "Nh": c.Nh},
        "cpu_baseline": {"value": value, "unit": "GS/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GS/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ----------------------------------------------------------------------------- main


DEFAULT_CONFIG = "C5"
DEFAULT_ALSO = ["C3"]
ALSO_KEYS = ("value", "unit", "ms_per_step", "ms_per_step_median", "ms_per_step_p20", "config", "roofline",
             "fp32", "metric_roofline", "e2e", "gpu_launches", "launch_mode", "clocks", "kernel", "plan_ms",
             "cpu_baseline", "page_comparison")


def workload(name: str, blocks: int = 0) -> W.Workload:
    """A workload by name; with blocks > 0 a single-call workload shortened to that many blocks."""
    w = W.WORKLOADS[name]
    if blocks > 0 and len(w.calls) == 1:
        w = dataclasses.replace(W.scaled(w, blocks),
                                description=f"{w.description}, shortened to k={blocks} blocks")
    return w


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(W.WORKLOADS) + sorted(W.CHANNELIZERS))
    ap.add_argument("--also", default=None,
                    help="comma-separated further workloads measured in the same run and reported under "
                         f"'also' (default: {','.join(DEFAULT_ALSO)} with the default workload, else none)")
    ap.add_argument("--dft-engine", choices=["fp32", "tensor"], default="fp32",
                    help="16-point DFTs as float32 butterflies (default) or on the tensor cores (N = 4096 and N >= 16384)")
    ap.add_argument("--blocks", type=int, default=0,
                    help="shorten a single-call workload to this many blocks (smaller profiler captures)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--direct", action="store_true",
                    help="launch each call from Python (per-launch events) instead of replaying a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.config in W.CHANNELIZERS:
        c = W.CHANNELIZERS[args.config]
        out = run_chan_reference(args, c, world, rank) if args.impl == "reference" else run_chan(
            args, c, world, rank, local)
    else:
        w = workload(args.config, args.blocks)
        if args.impl == "reference":
            out = run_reference(args, w, world, rank)
        else:
            out = run_ours(args, w, world, rank, local)
            also = DEFAULT_ALSO if args.also is None and args.config == DEFAULT_CONFIG else \
                [a for a in (args.also or "").split(",") if a]
            if also:
                out["also"] = []
                for name in also:
                    r = run_ours(args, workload(name, args.blocks), world, rank, local,
                                 cpu_budget=min(args.cpu_budget, 6.0))
                    out["also"].append({k: r[k] for k in ALSO_KEYS if k in r})
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
