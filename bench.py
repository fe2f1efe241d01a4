"""Benchmark of the GB300 addmm GEMM path (bf16 / MXFP4, persistent / Stream-K schedules).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--mode streamk] [--no-extras]

One step is one addmm of the workload (default: bf16 8192 x 8192 x 8192 with a bf16 bias,
bf16 output, Stream-K over all SMs).  Inputs are resident in HBM when the timed region starts;
A + B + C (384 MiB) exceed the 129 MB L2, so no flush is needed between steps.  Prints one JSON
line (rank 0).  Under torchrun every rank runs an independent replica on its own GPU (the GEMM
has no exchange step); the value is the sum of the ranks' work over the slowest rank's time.

--impl reference times the CPU oracle (plain binary64 C++ on the host cores) on a bounded
sample of the same workload: the comparison arm, not a target.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE_METRIC = "GEMM TFLOPS (bf16, MXFP4) per schedule and % of GB300 dense tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp4 dense peak relative to bf16 dense (nominal 13.5 / 2.25 PFLOP/s; MXFP4 with E8M0 scales
# runs at the fp4 rate)
FP4_OVER_BF16 = 13.5 / 2.25
# fp8 dense peak relative to bf16 dense (nominal 4.5 / 2.25 PFLOP/s)
FP8_OVER_BF16 = 4.5 / 2.25
FORMAT_CODE = {"bf16": 0, "mxfp4": 1, "fp8": 2}
# Nominal dense tensor peaks of one GB300 the targets are stated against (TFLOP/s): bf16
# ~2.25 PFLOP/s, fp8 4.5, FP4 ~9 PFLOP/s.
NOMINAL_DENSE_TFLOPS = {"bf16": 2250.0, "fp8": 4500.0, "mxfp4": 9000.0}
DTYPE_NAME = {"bf16": "bf16", "mxfp4": "mxfp4(e2m1+e8m0)", "fp8": "fp8(e4m3)"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="addmm_bf16_8192")
    ap.add_argument("--mode", default="streamk", choices=["dp", "persistent", "streamk", "hybrid", "auto"])
    ap.add_argument("--num-sms", type=int, default=0)
    ap.add_argument("--no-extras", action="store_true", help="skip the per-schedule extras")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end timing")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value, device=None):
    """Largest value over all ranks (the job's time is set by its slowest replica)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value, device=None):
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Sources outside the captured kernels' device code: the host API (its planning is checked
# separately, by comparing the recorded plan), the host-buffer copies, the no-allocation entry
# point and the backward's column sum.
NOT_IN_CAPTURED_LAUNCHES = {"sk_api.cu", "sk_host.cu", "sk_static.cu", "sk_reduce.cu"}


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sm_constrained_persistent_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in NOT_IN_CAPTURED_LAUNCHES:
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def plan_signature(plan):
    """The launch a plan makes: grid, CTAs per tile, tile and the Stream-K split."""
    return {"grid": plan.grid, "ctas_per_tile": plan.ctas_per_tile,
            "tile": f"{plan.tile_m}x{plan.tile_n}x{plan.tile_k}", "sk_tiles": plan.sk_tiles,
            "whole_tiles": plan.whole_tiles, "raster_group": plan.raster_group}


def recorded_traffic(kernel_key, plan=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel
    source and (when recorded) the same launch plan."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    entry = d.get("kernels", {}).get(kernel_key)
    if entry is None:
        return None
    if plan is not None and "plan" in entry and entry["plan"] != plan_signature(plan):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            mx = smax
            sms.append(sm)
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        load = [s for s in sms if s >= 0.5 * max(sms)]
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


def tile_efficiency(plan, sm_count, num_sms=0):
    """Tile-quantisation efficiency: useful k-iterations / (workers the call may use x the
    busiest worker's iterations).  Workers are SMs, or SM pairs for pair tiles; the call may
    use num_sms SMs (all when <= 0)."""
    import sm_constrained_persistent_gb300 as sk
    segs = sk.sk_plan_segments(plan)
    per_cta = np.zeros(plan.grid, dtype=np.int64)
    np.add.at(per_cta, segs[:, 0], segs[:, 3] - segs[:, 2])
    total = int(per_cta.sum())
    sms = sm_count if num_sms <= 0 or num_sms > sm_count else num_sms
    slots = max(1, sms // plan.ctas_per_tile)
    if plan.grid > slots:      # data-parallel: workers run in waves of one per slot
        per_slot = np.zeros(slots, dtype=np.int64)
        np.add.at(per_slot, np.arange(plan.grid) % slots, per_cta)
        return total / (slots * int(per_slot.max()))
    return total / (slots * int(per_cta.max()))


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------

class Problem:
    """Device-resident inputs and output of one workload, plus pinned host copies (for e2e)."""

    def __init__(self, name, device):
        import torch
        from sm_constrained_persistent_gb300 import inputs
        p = inputs.workload(name)
        self.name, self.p, self.device = name, p, device
        self.fmt, self.M, self.N, self.K = p["format"], p["M"], p["N"], p["K"]
        self.out_dtype = torch.bfloat16 if p["out_dtype"] == "bf16" else torch.float32

        def pinned(x, dtype=None):
            t = torch.from_numpy(np.ascontiguousarray(x))
            if dtype is not None:
                t = t.view(dtype)
            return t.pin_memory()

        if self.fmt == "bf16":
            self.host = {"A": pinned(p["A"].view(np.int16), torch.bfloat16),
                         "B": pinned(p["B"].view(np.int16), torch.bfloat16)}
        elif self.fmt == "fp8":
            self.host = {"A": pinned(p["A"]), "B": pinned(p["B"])}
        else:
            self.host = {"A": pinned(p["A"]), "A_scale": pinned(p["A_scale"]),
                         "B": pinned(p["B"]), "B_scale": pinned(p["B_scale"])}
        b = p["bias"]
        if b is not None:
            self.host["bias"] = pinned(b.view(np.int16), torch.bfloat16) if b.dtype == np.uint16 \
                else pinned(b)
        self.dev = {k: v.to(device) for k, v in self.host.items()}
        self.C = torch.empty((self.M, self.N), dtype=self.out_dtype, device=device)
        self.C_host = torch.empty((self.M, self.N), dtype=self.out_dtype).pin_memory()
        self.flops = 2.0 * self.M * self.N * self.K

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host.values())

    def d2h_bytes(self):
        return self.C.numel() * self.C.element_size()

    def call(self, mode, num_sms, stream_ptr, dev=None, options=None):
        """One addmm through the C ABI (the _ex form when options are given).  Returns the
        status code."""
        import sm_constrained_persistent_gb300 as sk
        d = self.dev if dev is None else dev
        bias = d["bias"].data_ptr() if "bias" in d else None
        od = sk.SK_BF16 if self.out_dtype.itemsize == 2 else sk.SK_F32
        m = sk.MODES[mode]
        if self.fmt == "bf16":
            if options is None:
                return sk.sk_gemm_bf16(d["A"].data_ptr(), d["B"].data_ptr(), bias,
                                       self.C.data_ptr(), od, self.M, self.N, self.K, num_sms, m,
                                       stream_ptr)
            return sk.sk_gemm_bf16_ex(d["A"].data_ptr(), d["B"].data_ptr(), bias,
                                      self.C.data_ptr(), od, self.M, self.N, self.K, num_sms, m,
                                      options, stream_ptr)
        if self.fmt == "fp8":
            if options is None:
                return sk.sk_gemm_fp8(d["A"].data_ptr(), d["B"].data_ptr(), bias,
                                      self.C.data_ptr(), od, self.M, self.N, self.K, num_sms, m,
                                      stream_ptr)
            return sk.sk_gemm_fp8_ex(d["A"].data_ptr(), d["B"].data_ptr(), bias,
                                     self.C.data_ptr(), od, self.M, self.N, self.K, num_sms, m,
                                     options, stream_ptr)
        if options is None:
            return sk.sk_gemm_mxfp4(d["A"].data_ptr(), d["A_scale"].data_ptr(), d["B"].data_ptr(),
                                    d["B_scale"].data_ptr(), bias, self.C.data_ptr(), od, self.M,
                                    self.N, self.K, num_sms, m, stream_ptr)
        return sk.sk_gemm_mxfp4_ex(d["A"].data_ptr(), d["A_scale"].data_ptr(), d["B"].data_ptr(),
                                   d["B_scale"].data_ptr(), bias, self.C.data_ptr(), od, self.M,
                                   self.N, self.K, num_sms, m, options, stream_ptr)

    def kernels_per_call(self):
        return 2 if self.fmt == "mxfp4" else 1   # MXFP4: the scale-layout kernel + the GEMM


L2_FLUSH_BYTES = 256 << 20   # twice the 129 MB L2


class L2Flush:
    """Evicts the operands from L2 between timed calls: a 256 MiB write (the eviction), then a
    256 MiB read of another buffer, so that the lines left in L2 are clean.  Without the read,
    the timed call would also pay for writing back the flush's own dirty lines."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.r = torch.ones((L2_FLUSH_BYTES // 4 // 1024, 1024), dtype=torch.float32, device=device)
        self.out = torch.empty(1024, dtype=torch.float32, device=device)

    def __call__(self):
        import torch
        self.w.fill_(1.0)
        torch.amax(self.r, dim=0, out=self.out)


def needs_flush(prob):
    """Operands that fit in L2 would stay there between steps: flush then."""
    operand_bytes = sum(t.numel() * t.element_size() for k, t in prob.dev.items() if k != "bias")
    return operand_bytes < L2_FLUSH_BYTES


def time_calls(prob, mode, num_sms, steps, warmup, dist=None, options=None, flush=None):
    """Device time of `steps` calls (after `warmup`), CUDA events on the launch stream,
    barrier + synchronize on both sides.  Back to back when the operands exceed L2; otherwise
    a 256 MiB write flushes L2 before each call and only the calls are timed.
    Returns (total ms of the calls, per-call ms list)."""
    import torch
    import sm_constrained_persistent_gb300 as sk
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    flush = needs_flush(prob) if flush is None else flush
    scrub = L2Flush(prob.device) if flush else None
    for _ in range(warmup):
        st = prob.call(mode, num_sms, sp, options=options)
        if st != 0:
            raise RuntimeError(f"warm-up call failed: {sk.STATUS.get(st, st)}")
    torch.cuda.synchronize()
    if sk.sk_stream_status(sp) != 0:
        raise RuntimeError("kernel reported an error during warm-up")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(dist)
    torch.cuda.synchronize()
    for s, e in ev:
        if flush:
            scrub()
        s.record(stream)
        prob.call(mode, num_sms, sp, options=options)
        e.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    if sk.sk_stream_status(sp) != 0:
        raise RuntimeError("kernel reported an error in the timed region")
    per = [s.elapsed_time(e) for s, e in ev]
    total = sum(per) if flush else ev[0][0].elapsed_time(ev[-1][1])
    return total, per


def time_e2e(prob, mode, num_sms, steps, warmup):
    """Same metric end to end through the host-buffer C-ABI call: every step copies the
    step's inputs from pinned host memory to the device, computes, and copies C back to
    pinned host memory (the library overlaps the three in row blocks), all inside the timed
    region.  Returns ms per step."""
    import torch
    import sm_constrained_persistent_gb300 as sk
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    h = prob.host
    bias = h["bias"].data_ptr() if "bias" in h else None
    od = sk.SK_BF16 if prob.out_dtype.itemsize == 2 else sk.SK_F32
    m = sk.MODES[mode]

    def one():
        if prob.fmt == "bf16":
            st = sk.sk_gemm_bf16_host(h["A"].data_ptr(), h["B"].data_ptr(), bias,
                                      prob.C_host.data_ptr(), od, prob.M, prob.N, prob.K,
                                      num_sms, m, None, sp)
        elif prob.fmt == "fp8":
            st = sk.sk_gemm_fp8_host(h["A"].data_ptr(), h["B"].data_ptr(), bias,
                                     prob.C_host.data_ptr(), od, prob.M, prob.N, prob.K,
                                     num_sms, m, None, sp)
        else:
            st = sk.sk_gemm_mxfp4_host(h["A"].data_ptr(), h["A_scale"].data_ptr(),
                                       h["B"].data_ptr(), h["B_scale"].data_ptr(), bias,
                                       prob.C_host.data_ptr(), od, prob.M, prob.N, prob.K,
                                       num_sms, m, None, sp)
        if st != 0:
            raise RuntimeError(f"host-buffer call failed: {sk.STATUS.get(st, st)}")

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        one()
    e.record(stream)
    torch.cuda.synchronize()
    if sk.sk_stream_status(sp) != 0:
        raise RuntimeError("kernel reported an error in the end-to-end region")
    return s.elapsed_time(e) / steps


def cpu_baseline(prob, seconds):
    """The oracle, as it stands, on a block of rows of the same workload (about `seconds` of
    host time).  Returns the cpu_baseline object in the metric's unit."""
    import oracle
    p = prob.p
    threads = oracle.hardware_threads()

    def run(rows):
        t0 = time.perf_counter()
        if prob.fmt == "bf16":
            oracle.addmm_bf16(p["A"], p["B"], p["bias"], rows=(0, rows), threads=threads)
        elif prob.fmt == "fp8":
            oracle.addmm_fp8(p["A"], p["B"], p["bias"], rows=(0, rows), threads=threads)
        else:
            oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"],
                               rows=(0, rows), threads=threads)
        return time.perf_counter() - t0

    # two probes: a tiny one, then one of about a tenth of the budget, to estimate the rate
    probe_rows = min(prob.M, max(threads, 8))
    t_probe = run(probe_rows)
    probe_rows = int(min(prob.M, max(probe_rows, probe_rows * 0.1 * seconds / max(t_probe, 1e-3))))
    t_probe = run(probe_rows)
    rows = int(min(prob.M, max(probe_rows, probe_rows * seconds / max(t_probe, 1e-3))))
    rows = max(threads, rows - rows % threads) if rows >= threads else rows
    t = run(rows)
    flops = 2.0 * rows * prob.N * prob.K
    return {"value": flops / t / 1e12, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
            "sample": f"rows [0, {rows}) of the {prob.M}x{prob.N}x{prob.K} {prob.fmt} addmm "
                      f"({flops / 1e9:.1f} GFLOP, {t:.1f} s, binary64 accumulation)"}


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    import __graft_entry__
    __graft_entry__.build()          # no-op when the library is up to date
    import sm_constrained_persistent_gb300 as sk

    props = torch.cuda.get_device_properties(local)
    sm_count = props.multi_processor_count
    prob = Problem(args.workload, device)
    torch.cuda.synchronize()

    with ClockSampler(local) as clocks:
        total_ms, per = time_calls(prob, args.mode, args.num_sms, args.steps, args.warmup, dist)
    ms_max = max_over_ranks(dist, total_ms / args.steps, device)
    flops_all = sum_over_ranks(dist, prob.flops * args.steps, device)
    value = flops_all / (ms_max * args.steps * 1e-3) / 1e12
    clock = clocks.summary()

    plan = sk.sk_plan(FORMAT_CODE[prob.fmt], prob.M, prob.N, prob.K, args.num_sms,
                      args.mode, sm_count)
    peaks, peak_src = measured_peaks()
    bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    if prob.fmt == "bf16":
        peak, peak_note = bf16_peak, f"bf16 dense, burst, {peak_src}"
    elif prob.fmt == "fp8":
        peak = bf16_peak * FP8_OVER_BF16
        peak_note = f"fp8 dense = {peak_src} bf16 burst x {FP8_OVER_BF16:g} (nominal ratio)"
    else:
        peak = bf16_peak * FP4_OVER_BF16
        peak_note = f"fp4 dense = {peak_src} bf16 burst x {FP4_OVER_BF16:g} (nominal ratio)"
    gemm_ms = statistics.mean(per)   # one GEMM kernel dominates each call
    kernel_key = (f"gemm<{prob.fmt},{plan.tile_m}x{plan.tile_n}>"
                  f":{args.workload}:{args.mode}")
    # Algorithmic bytes: every operand (and scale and bias) read once, C written once.
    alg_bytes = sum(t.numel() * t.element_size() for t in prob.dev.values()) + prob.d2h_bytes()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ridge = peak * 1e12 / (hbm * 1e9)                     # flop per byte
    if prob.flops / alg_bytes < ridge:                    # below the ridge: HBM-bound
        achieved = alg_bytes / (gemm_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": round(hbm, 1),
                    "unit": "GB/s", "frac": round(achieved / hbm, 4),
                    "traffic": recorded_traffic(kernel_key, plan),
                    "peak_source": f"copy bandwidth, {peak_src}", "kernel": kernel_key,
                    "algorithmic_bytes": alg_bytes}
    else:
        achieved = prob.flops / (gemm_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "traffic": recorded_traffic(kernel_key, plan), "peak_source": peak_note,
                    "kernel": kernel_key, "algorithmic_flops": prob.flops}

    e2e = None
    if not args.no_e2e:
        e2e_ms = time_e2e(prob, args.mode, args.num_sms, max(3, min(args.steps, 10)), 2)
        e2e_ms_max = max_over_ranks(dist, e2e_ms, device)
        e2e = {"value": round(sum_over_ranks(dist, prob.flops, device) / (e2e_ms_max * 1e-3) / 1e12, 2),
               "unit": "TFLOPS", "h2d_bytes_per_step": prob.h2d_bytes(),
               "d2h_bytes_per_step": prob.d2h_bytes(),
               "call": f"sk_gemm_{prob.fmt}_host (pinned host buffers; copies overlapped with "
                       "the GEMM in row blocks)"}

    result = {
        "metric": HEADLINE_METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_NAME[prob.fmt], "data": "synthetic",
        "config": {"workload": args.workload, "M": prob.M, "N": prob.N, "K": prob.K,
                   "format": prob.fmt, "out": str(prob.out_dtype).replace("torch.", ""),
                   "bias": prob.p["bias"] is not None, "mode": args.mode,
                   "num_sms": args.num_sms if args.num_sms > 0 else sm_count,
                   "grid": plan.grid, "tile": f"{plan.tile_m}x{plan.tile_n}x{plan.tile_k}",
                   "tile_quant_eff": round(tile_efficiency(plan, sm_count, args.num_sms), 4),
                   "pct_of_measured_peak": round(100 * value / world / peak, 2),
                   "pct_of_nominal_peak": round(100 * value / world / NOMINAL_DENSE_TFLOPS[prob.fmt], 2),
                   "l2": ("L2 flushed before each step (256 MiB write, then a 256 MiB read so "
                          "the lines left are clean)" if needs_flush(prob)
                          else "inputs larger than L2 (no flush)"),
                   "parallelism": f"replicas{world}"},
        "roofline": roofline, "e2e": e2e,
        "gpu_launches": args.steps * prob.kernels_per_call(),
        "clocks": {"sm_mhz": clock["sm_mhz"], "sm_max_mhz": clock["sm_max_mhz"],
                   "reasons": clock["reasons"]},
    }
    if not args.no_extras:
        result["extras"] = extras(prob, sm_count, dist)
    if world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(prob, args.cpu_seconds)
    # last key: the per-config, per-schedule figures in a form short enough to survive a
    # truncated log tail
    result["summary"] = summary_block(result, args.mode, prob.fmt, peak)
    if rank == 0:
        print(json.dumps(result, separators=(",", ":")), flush=True)
    if dist is not None:
        dist.destroy_process_group()


MODE_KEY = {"dp": "dp", "persistent": "pe", "streamk": "sk", "hybrid": "hy", "auto": "au"}


def summary_block(result, mode, fmt, measured_peak):
    """Compact per-config x schedule table: [ms, TFLOPS, % of nominal dense peak, % of measured
    peak, tile-quantisation efficiency] per schedule (dp, pe = persistent, sk = Stream-K,
    hy = hybrid); the num_sms sweeps as [ms, TFLOPS or GB/s, SMs used]."""
    peaks, _ = measured_peaks()
    bpeak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    meas = {"bf16": bpeak, "fp8": bpeak * FP8_OVER_BF16, "mxfp4": bpeak * FP4_OVER_BF16}

    def row(r, f):
        t = r["tflops"]
        return [r["ms"], round(t), round(100 * t / NOMINAL_DENSE_TFLOPS[f], 1),
                round(100 * t / meas[f], 1), r["tile_quant_eff"]]

    def table(rows, f):
        return {MODE_KEY.get(m, m): row(r, f) for m, r in rows.items()}

    out = {"cols": "ms,TFLOPS,%nominal,%measured,tile_quant_eff",
           "nominal_tf": {"bf16": 2250, "fp8": 4500, "mxfp4": 9000},
           "measured_tf": {k: round(v, 1) for k, v in meas.items()}}
    cfg = result["config"]
    out["headline"] = {"workload": cfg["workload"], MODE_KEY[mode]: row(
        {"ms": result["ms_per_step"], "tflops": result["value"],
         "tile_quant_eff": cfg["tile_quant_eff"]}, fmt)}
    ex = result.get("extras")
    if not ex:
        return out
    # the num_sms sweeps first and the per-schedule tables of the headline formats last, so a
    # log cut from the front keeps the MXFP4 and wave-quantised rows
    sw = ex.get("num_sms_sweep_persistent", {})
    if "gemm_bf16_4096" in sw:
        out["c4_4096_pe"] = {ns: [r["ms"], round(r["tflops"]), r.get("sms_used")]
                             for ns, r in sw["gemm_bf16_4096"].items()}
    if "gemm_bf16_skinny_64x14336x4096" in sw:
        out["c4_skinny_pe_gbs"] = {ns: [r["ms"], round(r["gbs"]), r.get("sms_used")]
                                   for ns, r in sw["gemm_bf16_skinny_64x14336x4096"].items()}
    names = [("c0_bf16_256x256x512_f32", "addmm_bf16_256x256x512_f32out", "bf16"),
             ("bf16_1024x1024x16384", "gemm_bf16_1024x1024x16384", "bf16"),
             ("fp8_8192", "addmm_fp8_8192", "fp8"),
             ("c1_bf16_8192", "addmm_bf16_8192", "bf16")]
    for key, name, f in names:
        if name in ex:
            out[key] = table(ex[name], f)
    wq = ex.get("gemm_bf16_1920x1920x16384", {})
    if wq:
        out["c2_1920_tile128"] = table(wq["tile_128x128"], "bf16")
        out["c2_1920_auto"] = table(wq["auto"], "bf16")
    if "addmm_mxfp4_8192" in ex:
        out["c3_mxfp4_8192"] = table(ex["addmm_mxfp4_8192"], "mxfp4")
    return out


def sms_used(pr, mode, num_sms, sm_count, options=None):
    """Distinct SMs one call ran on, from the kernels' SM-usage record (an untimed call)."""
    import torch
    import sm_constrained_persistent_gb300 as sk
    opts = dict(options or {})
    plan = sk.sk_plan(FORMAT_CODE[pr.fmt], pr.M, pr.N, pr.K, num_sms, mode, sm_count, opts)
    ctas = plan.grid * plan.ctas_per_tile
    record = torch.full((ctas,), -1, dtype=torch.int32, device=pr.device)
    opts.update(sm_record=record.data_ptr(), sm_record_len=ctas)
    stream = torch.cuda.current_stream()
    if pr.call(mode, num_sms, stream.cuda_stream, options=opts) != 0:
        raise RuntimeError("recorded call failed")
    torch.cuda.synchronize()
    if sk.sk_stream_status(stream.cuda_stream) != 0:
        raise RuntimeError("recorded call reported an error")
    r = record.cpu().numpy()
    if (r < 0).any():
        raise RuntimeError("a CTA did not record its SM")
    return int(len(np.unique(r)))


def _time_modes(pr, modes, sm_count, peak, dist, num_sms=0, options=None, steps=10, warmup=3,
                flush=None):
    """ms, TFLOPS, % of peak, grid, tile and tile-quantisation efficiency per mode."""
    import sm_constrained_persistent_gb300 as sk
    res = {}
    for mode in modes:
        total, _ = time_calls(pr, mode, num_sms, steps, warmup, dist, options, flush)
        ms = total / steps
        plan = sk.sk_plan(FORMAT_CODE[pr.fmt], pr.M, pr.N, pr.K, num_sms, mode, sm_count,
                          options)
        tflops = pr.flops / (ms * 1e-3) / 1e12
        res[mode] = {"ms": round(ms, 4), "tflops": round(tflops, 1),
                     "pct_peak": round(100 * tflops / peak, 1), "grid": plan.grid,
                     "ctas": plan.grid * plan.ctas_per_tile,
                     "tile": f"{plan.tile_m}x{plan.tile_n}x{plan.tile_k}",
                     "tile_quant_eff": round(tile_efficiency(plan, sm_count, num_sms), 4)}
    return res


def corun(pr, sm_count, gemm_calls=5, copy_bytes=256 << 20):
    """The SM-constrained GEMM (persistent and Stream-K on half the SMs) beside a memory-bound
    copy on a second stream: each stream's throughput alone and together (events per stream).
    This is the intra-device sharing the num_sms cap exists for."""
    import torch
    half = sm_count // 2
    src = torch.ones(copy_bytes // 4, dtype=torch.float32, device=pr.device)
    dst = torch.empty_like(src)
    s_gemm, s_copy = torch.cuda.Stream(), torch.cuda.Stream()

    def run(do_gemm, do_copy, mode, copies):
        ev = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for k in ("gemm", "copy")}
        torch.cuda.synchronize()
        if do_copy:
            with torch.cuda.stream(s_copy):
                ev["copy"][0].record(s_copy)
                for _ in range(copies):
                    dst.copy_(src)
                ev["copy"][1].record(s_copy)
        if do_gemm:
            with torch.cuda.stream(s_gemm):
                ev["gemm"][0].record(s_gemm)
                for _ in range(gemm_calls):
                    pr.call(mode, half, s_gemm.cuda_stream)
                ev["gemm"][1].record(s_gemm)
        torch.cuda.synchronize()
        res = {}
        if do_gemm:
            ms = ev["gemm"][0].elapsed_time(ev["gemm"][1]) / gemm_calls
            res["gemm_tflops"] = round(pr.flops / (ms * 1e-3) / 1e12, 1)
        if do_copy:
            ms = ev["copy"][0].elapsed_time(ev["copy"][1]) / copies
            res["copy_gbs"] = round(2 * copy_bytes / (ms * 1e-3) / 1e9, 1)
        return res

    out = {"num_sms": half, "copy": f"{copy_bytes >> 20} MiB device-to-device copies"}
    for mode in ("persistent", "streamk"):
        run(True, False, mode, 0)                               # warm-up
        alone = run(True, False, mode, 0)
        gemm_ms = pr.flops / (alone["gemm_tflops"] * 1e12) * 1e3 * gemm_calls
        copy_alone = run(False, True, mode, 20)
        per_copy_ms = 2 * copy_bytes / (copy_alone["copy_gbs"] * 1e9) * 1e3
        copies = max(4, int(gemm_ms / per_copy_ms))             # both streams busy as long
        both = run(True, True, mode, copies)
        out[mode] = {"gemm_alone_tflops": alone["gemm_tflops"],
                     "copy_alone_gbs": copy_alone["copy_gbs"],
                     "gemm_corun_tflops": both["gemm_tflops"], "copy_corun_gbs": both["copy_gbs"]}
    assert_ok = __import__("sm_constrained_persistent_gb300").sk_stream_status(s_gemm.cuda_stream)
    if assert_ok != 0:
        raise RuntimeError("co-run GEMM reported an error")
    return out


def backward(pr, bf16_peak, steps=10, warmup=3):
    """The addmm backward of the 8192^3 workload (dA = dC B^T, dB = A^T dC, dbias), bf16
    gradients, Stream-K: 4 M N K FLOPs per call (the column sum is not counted)."""
    import torch
    import sm_constrained_persistent_gb300 as sk
    M, N, K = pr.M, pr.N, pr.K
    dc = torch.randn((M, N), device=pr.device).to(torch.bfloat16)
    a, b = pr.dev["A"], pr.dev["B"]
    da = torch.empty((M, K), dtype=torch.bfloat16, device=pr.device)
    db = torch.empty((K, N), dtype=torch.bfloat16, device=pr.device)
    dbias = torch.empty((N,), dtype=torch.bfloat16, device=pr.device)
    stream = torch.cuda.current_stream()

    def call(mode):
        return sk.sk_addmm_backward_bf16(dc.data_ptr(), a.data_ptr(), b.data_ptr(), da.data_ptr(),
                                         db.data_ptr(), dbias.data_ptr(), sk.SK_BF16, M, N, K, 0,
                                         sk.MODES[mode], stream.cuda_stream)

    res = {}
    for mode in ("streamk", "hybrid"):
        for _ in range(warmup):
            if call(mode) != 0:
                raise RuntimeError("backward call failed")
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(steps):
            call(mode)
        e.record(stream)
        torch.cuda.synchronize()
        if sk.sk_stream_status(stream.cuda_stream) != 0:
            raise RuntimeError("backward reported an error")
        ms = s.elapsed_time(e) / steps
        tflops = 4.0 * M * N * K / (ms * 1e-3) / 1e12
        res[mode] = {"ms": round(ms, 4), "tflops": round(tflops, 1),
                     "pct_peak": round(100 * tflops / bf16_peak, 1)}
    return res


# Shapes outside the set the automatic choice's cost model was fitted on.
AUTO_CHECK_SHAPES = [(3584, 3584, 3584), (1280, 5120, 5120), (640, 2560, 16384),
                     (7168, 7168, 1536), (96, 8192, 8192), (4864, 1792, 8192)]


def auto_selection(device, sm_count, bpeak, dist):
    """SK_MODE_AUTO against every schedule x tile kind on shapes held out of its calibration:
    the automatic plan's time, the fastest configuration and the ratio."""
    from sm_constrained_persistent_gb300 import inputs
    tiles = {"pair": {"tile_m": 256}, "128x256": {"tile_m": 128, "tile_n": 256},
             "128x128": {"tile_m": 128, "tile_n": 128}, "128x96": {"tile_m": 128, "tile_n": 96}}
    res = {}
    for (M, N, K) in AUTO_CHECK_SHAPES:
        name = f"gemm_bf16_{M}x{N}x{K}"
        inputs.WORKLOADS.setdefault(name, ("bf16", M, N, K, dict(operand_scale="sqrt_k",
                                                                 bias="none"), "bf16", 1240))
        pr = Problem(name, device)
        auto = _time_modes(pr, ["auto"], sm_count, bpeak, dist)["auto"]
        best = None
        for tname, opt in tiles.items():
            if (tname == "pair" and M <= 128) or (tname == "128x96" and M > 128):
                continue
            for mode, r in _time_modes(pr, ["dp", "persistent", "streamk", "hybrid"], sm_count,
                                       bpeak, dist, options=opt).items():
                if best is None or r["ms"] < best["ms"]:
                    best = dict(r, mode=mode)
        # the measured choice: sk_autotune on this problem, then auto mode again
        import sm_constrained_persistent_gb300 as sk
        d = pr.dev
        sk.autotune("bf16", d["A"], d["B"], d.get("bias"), out=pr.C, reps=5)
        tuned = _time_modes(pr, ["auto"], sm_count, bpeak, dist)["auto"]
        res[name] = {"auto_ms": auto["ms"], "auto_tile": auto["tile"], "best_ms": best["ms"],
                     "best": f"{best['mode']} {best['tile']}",
                     "auto_over_best": round(auto["ms"] / best["ms"], 3),
                     "autotuned_ms": tuned["ms"],
                     "autotuned_over_best": round(tuned["ms"] / best["ms"], 3)}
        del pr
    return res


def extras(prob, sm_count, dist):
    """Per-schedule throughput of the benchmark workloads, each timed on its own after the
    headline region (3 warm-up + 10 timed calls per entry), and the SM-constrained sweep."""
    import torch
    out = {}
    peaks, _ = measured_peaks()
    bpeak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    modes = ["dp", "persistent", "streamk", "hybrid"]
    cache = {prob.name: prob}

    def get(name):
        if name not in cache:
            cache[name] = Problem(name, prob.device)
        return cache[name]

    # the 256 x 256 x 512 fp32-output addmm: data-parallel, and Stream-K over 3 CTAs
    pr = get("addmm_bf16_256x256x512_f32out")
    out[pr.name] = _time_modes(pr, ["dp"], sm_count, bpeak, dist)
    out[pr.name]["sk3"] = _time_modes(pr, ["streamk"], sm_count, bpeak, dist, num_sms=3)["streamk"]
    for name in ["addmm_bf16_8192", "addmm_mxfp4_8192", "addmm_fp8_8192",
                 "gemm_bf16_1024x1024x16384"]:
        pr = get(name)
        peak = bpeak * {"bf16": 1.0, "mxfp4": FP4_OVER_BF16, "fp8": FP8_OVER_BF16}[pr.fmt]
        out[name] = _time_modes(pr, modes, sm_count, peak, dist)
    # the wave-quantised shape: its stated 128x128 tiles (225 tiles) and the automatic choice
    pr = get("gemm_bf16_1920x1920x16384")
    out["gemm_bf16_1920x1920x16384"] = {
        "tile_128x128": _time_modes(pr, modes, sm_count, bpeak, dist,
                                    options={"tile_m": 128, "tile_n": 128}),
        "auto": _time_modes(pr, modes, sm_count, bpeak, dist)}
    # SM-constrained persistent sweep: time and TFLOPS per num_sms
    sweep = {}
    for name in ["gemm_bf16_4096", "gemm_bf16_skinny_64x14336x4096"]:
        pr = get(name)
        rows = {}
        for ns in [1, 16, 32, 64, 128, sm_count]:
            r = _time_modes(pr, ["persistent"], sm_count, bpeak, dist, num_sms=ns,
                            steps=5 if ns < 16 else 10, warmup=2)["persistent"]
            r["tflops_per_sm"] = round(r["tflops"] / ns, 2)
            r["sms_used"] = sms_used(pr, "persistent", ns, sm_count)
            if "skinny" in name:
                bytes_moved = sum(t.numel() * t.element_size() for t in pr.dev.values()) + \
                    pr.C.numel() * pr.C.element_size()
                r["gbs"] = round(bytes_moved / (r["ms"] * 1e-3) / 1e9, 1)
                r["pct_hbm"] = round(100 * r["gbs"] / hbm, 1)
            rows[str(ns)] = r
        sweep[name] = rows
    out["num_sms_sweep_persistent"] = sweep
    # warm L2 (operands left in L2 by the previous call) against the flushed numbers above
    warm = {}
    for name, opt in [("gemm_bf16_1920x1920x16384", {"tile_m": 128, "tile_n": 128}),
                      ("gemm_bf16_skinny_64x14336x4096", None)]:
        pr = get(name)
        cold = _time_modes(pr, ["persistent", "streamk"], sm_count, bpeak, dist, options=opt)
        hot = _time_modes(pr, ["persistent", "streamk"], sm_count, bpeak, dist, options=opt,
                          flush=False)
        warm[name] = {m: {"cold_ms": cold[m]["ms"], "warm_ms": hot[m]["ms"]} for m in cold}
    out["l2_warm_vs_cold"] = warm
    out["auto_selection"] = auto_selection(prob.device, sm_count, bpeak, dist)
    out["corun_half_sms"] = corun(get("addmm_bf16_8192"), sm_count)
    out["addmm_backward_bf16_8192"] = backward(get("addmm_bf16_8192"), bpeak)
    for name in list(cache):
        if cache[name] is not prob:
            del cache[name]
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return
    import oracle
    from sm_constrained_persistent_gb300 import inputs
    p = inputs.workload(args.workload)
    threads = oracle.hardware_threads()
    rows = max(threads, 16)
    M, N, K = p["M"], p["N"], p["K"]

    def step():
        if p["format"] == "bf16":
            oracle.addmm_bf16(p["A"], p["B"], p["bias"], rows=(0, rows), threads=threads)
        elif p["format"] == "fp8":
            oracle.addmm_fp8(p["A"], p["B"], p["bias"], rows=(0, rows), threads=threads)
        else:
            oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"],
                               rows=(0, rows), threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    flops = 2.0 * rows * N * K
    value = flops / dt / 1e12
    sample = (f"rows [0, {rows}) of the {M}x{N}x{K} {p['format']} addmm per step "
              f"({flops / 1e9:.2f} GFLOP), binary64 accumulation")
    print(json.dumps({
        "impl": "reference", "metric": HEADLINE_METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K, "format": p["format"],
                   "mode": args.mode},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
