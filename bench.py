"""Benchmark: bin + forward + backward per iteration on the 800x800, 409,660-splat
Lego-shaped synthetic set (seed 3), one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--config NAME]

GPU arm: inputs resident in HBM, warm arena, L2 flushed (256 MB write) between
timed steps, each step bracketed by CUDA events on the launching stream, per
stage (bin / forward / backward) events as well.  e2e: the same steps with the
inputs copied from pinned host memory and the gradients and image copied back
inside the timed region.  N > 1 (torchrun): independent replicas, one per
GPU, the slowest rank's time counts.

Reference arm (--impl reference): the CPU oracle, unchanged, on the host
cores, on the same workload; each step is the whole frame cut into one band of
tile rows per core (each band bins every splat against its rows, then runs the
forward and backward), the bands in parallel worker processes, timed by the
wall clock.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gen  # noqa: E402

METRIC = "rasterize bin+fwd+bwd ms/iter @800×800, 409,660 splats; % of roofline"
FLUSH_BYTES = 256 << 20
# Lanes per SM per clock of the FP32 (FFMA) pipe and of the SFU's ex2: the
# formula the measured rates (peak_kernel) are shown beside.  GB300's SFU runs
# ex2 at 32 lanes per SM per clock (measured with gsr_peak_kernel).
FP32_LANES_PER_SM = 128
SFU_LANES_PER_SM = 32

# Algorithmic FP32 operations per unit (the counts come from the oracle's counters).
#   forward, per examined (pixel, splat): dx, dy, 5 for sigma, 2 range compares   = 9
#            per sigma-in-range evaluation: exponent scale, o*e, min, alpha cut    = 4  (+1 SFU exp)
#            per composited splat: 1-alpha, T(1-alpha), stop test, alpha*T, 3 FMA = 7
#   backward, per replayed (pixel, splat) below last_contributor                  = 9
#            per sigma-in-range evaluation                                          = 4  (+1 SFU exp)
#            per composited splat: 1/(1-alpha) (+1 SFU), T_j, alpha T_j, 3 rgb grads,
#            dL/dalpha (9), S update (3), clamp select, dL/dcolor_a, dL/dsigma,
#            5 conic/mean grads (12), and the 9 additions that accumulate them   = 44
FWD_OPS = {"n_eval": 9, "n_exp": 4, "n_contrib": 7}
BWD_OPS = {"n_eval": 9, "n_exp": 4, "n_contrib": 44}

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch, from one
# ncu capture (profiles/k_*.md), with the SHA-256 of the kernel sources it was
# taken on.  Once the sources change, the figure no longer describes the kernel
# and is reported as null.
RASTER_SOURCES = ("gaussian_splatting_tile_bin_gb300/csrc/raster.cu",
                  "gaussian_splatting_tile_bin_gb300/csrc/internal.cuh")
PROJECT_SOURCES = ("gaussian_splatting_tile_bin_gb300/csrc/project.cu",
                   "gaussian_splatting_tile_bin_gb300/csrc/internal.cuh")
RASTER_SHA256 = "01ed77677abb61440974f4d52d7aa690e31651757e8d5622f336866995f58d85"
PROJECT_SHA256 = "175bb9e55f6c1b3360e8b68de16750f83fbafe5efbb2c04b03160fcf883f5192"
NCU_TRAFFIC = {
    "forward": {"bytes": 22_278_144 + 120_576, "workload": "lego_final", "sources": RASTER_SOURCES,
                "sha256": RASTER_SHA256},
    "backward": {"bytes": 49_740_032 + 68_352, "workload": "lego_final", "sources": RASTER_SOURCES,
                 "sha256": RASTER_SHA256},
    "project_forward": {"bytes": 22_960_128 + 1_024, "workload": "lego_scene", "sources": PROJECT_SOURCES,
                        "sha256": PROJECT_SHA256},
    "project_backward": {"bytes": 37_718_528 + 136_960, "workload": "lego_scene", "sources": PROJECT_SOURCES,
                         "sha256": PROJECT_SHA256},
}


def sources_digest(sources) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(hashlib.sha256(f.read()).digest())
    return h.hexdigest()


def ncu_traffic(kind: str, workload: str):
    entry = NCU_TRAFFIC.get(kind)
    if entry is None or entry["workload"] != workload or sources_digest(entry["sources"]) != entry["sha256"]:
        return None
    return entry["bytes"]


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="gsr", choices=["gsr", "reference"])
    p.add_argument("--config", default="lego_final", choices=sorted(gen.CONFIGS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-cpu-all-cores", action="store_true",
                   help="skip the oracle's run on all host cores (tile-row bands in parallel processes)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--deterministic", action="store_true",
                   help="time the backward's deterministic mode (fixed-point accumulation)")
    p.add_argument("--bwd-per-splat", action="store_true",
                   help="time the backward's transposed (per-splat) loop nest instead of the per-pixel one")
    p.add_argument("--graph", action="store_true",
                   help="also time the whole step (binning, forward, backward) replayed as one captured CUDA graph")
    p.add_argument("--no-split", action="store_true",
                   help="run forward and backward as one CTA per tile (no chunks or segments of long lists)")
    p.add_argument("--split-forward", action="store_true",
                   help="split the forward's crowded lists too (GSR_OPT_SPLIT_FORWARD)")
    p.add_argument("--reserved", action="store_true",
                   help="time the step with the binning of a context that has a reservation (no host read-back) "
                        "instead of the default binning, which reads the pair count back every call")
    p.add_argument("--no-other-configs", action="store_true",
                   help="skip the lines of the other frames timed beside the headline one")
    p.add_argument("--no-projection", action="store_true",
                   help="skip the separate timing of the projection kernels")
    p.add_argument("--no-alu-peaks", action="store_true",
                   help="skip the FP32/SFU rate kernels (profiling runs; the roofline is then not reported)")
    p.add_argument("--min-warm-s", type=float, default=1.5,
                   help="keep warming up until this many seconds passed (clock sampling)")
    return p.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max over ranks (a scalar timing exchange, not a data-path collective)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_ms_per_iter(local_ms_sum: float, steps: int, world: int, device=None) -> float:
    """Whole-job ms per iteration: every rank runs `steps` iterations of its own
    replica, so the job finishes world x steps iterations in the slowest rank's
    time."""
    return reduce_max(local_ms_sum, world, device) / (steps * world)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0, "source": "fallback"}


def workload_label(wl):
    return f"{wl.name}: {wl.width}x{wl.height}, {wl.n:,} Splat2D, seed {wl.recipe.get('seed')}"


# --------------------------------------------------------------------------
# Clock sampling
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "sm_max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else None,
                             "hw_slowdown": parts[5], "hw_thermal": parts[6],
                             "sw_thermal": parts[7], "sw_power_cap": parts[8]})
            except ValueError:
                continue
        return rows

    @staticmethod
    def summarize(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r["power"] is None or r["power"] > 0] or rows
        reasons = []
        for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in loaded):
                reasons.append(name)
        return {"sm_mhz": float(np.median([r["sm"] for r in loaded])),
                "sm_max_mhz": float(max(r["sm_max"] for r in loaded)),
                "reasons": reasons, "samples": len(loaded)}


# --------------------------------------------------------------------------
# CPU oracle (the cpu_baseline leg and the reference arm)
# --------------------------------------------------------------------------

def cpu_baseline(wl):
    """The oracle, as it stands, on the whole workload once: binning, forward,
    backward.  Returns the timing and the oracle's evaluation counters."""
    import oracle
    t0 = time.perf_counter()
    keys, idx, ranges = oracle.bin_splats(wl.splats, wl.depths, wl.width, wl.height)
    t1 = time.perf_counter()
    f = oracle.forward(wl.splats, idx, ranges, wl.width, wl.height)
    t2 = time.perf_counter()
    b = oracle.backward(wl.splats, idx, ranges, wl.width, wl.height, wl.dl_dout)
    t3 = time.perf_counter()
    return {"ms": (t3 - t0) * 1e3, "bin_ms": (t1 - t0) * 1e3, "fwd_ms": (t2 - t1) * 1e3,
            "bwd_ms": (t3 - t2) * 1e3, "pairs": int(len(keys)),
            "fwd_counters": f["counters"], "bwd_counters": b["counters"]}


def _oracle_band(job):
    """One tile-row band of a workload through the oracle (bin, forward,
    backward); runs in a spawned worker process."""
    name, band, bands = job
    import oracle
    sub, _ = band_workload(gen.make(name), band, bands)
    keys, idx, ranges = oracle.bin_splats(sub.splats, sub.depths, sub.width, sub.height)
    oracle.forward(sub.splats, idx, ranges, sub.width, sub.height)
    oracle.backward(sub.splats, idx, ranges, sub.width, sub.height, sub.dl_dout)
    return len(keys)


def cpu_baseline_all_cores(name):
    """The oracle, as it stands, over the whole frame split into one tile-row
    band per host core, the bands in parallel worker processes (spawned: this
    process has used the GPU).  Returns (ms, cores)."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    cores = len(os.sched_getaffinity(0))
    # A worker that dies raises BrokenProcessPool here instead of hanging.
    with ProcessPoolExecutor(cores, mp_context=mp.get_context("spawn")) as pool:
        list(pool.map(_oracle_band, [(name, 0, cores)] * cores))   # workers up, oracle loaded
        t0 = time.perf_counter()
        list(pool.map(_oracle_band, [(name, k, cores) for k in range(cores)]))
        ms = (time.perf_counter() - t0) * 1e3
    return ms, cores


def band_workload(wl, band, bands):
    """Tile-row band `band` of `bands` as its own image (means shifted up)."""
    tiles_y = (wl.height + 15) // 16
    per = (tiles_y + bands - 1) // bands
    y0 = min(band * per, tiles_y) * 16
    y1 = min((band + 1) * per * 16, wl.height)
    s = wl.splats.copy()
    s[:, 1] -= np.float32(y0)
    dl = wl.dl_dout.reshape(wl.height, wl.width, 4)[y0:y1].reshape(-1, 4)
    return gen.from_arrays(f"{wl.name}[rows {y0}:{y1}]", wl.width, y1 - y0, s, wl.depths, dl), y1 - y0


def long_lists_label(args) -> str:
    if args.no_split:
        return "one CTA per tile"
    bwd = "backward: segments of tiles above a CTA slot's share of the work"
    if args.split_forward:
        return "forward: 512-position chunks past a head of max(1024, half the pairs per CTA slot); " + bwd
    return "forward: one CTA per tile; " + bwd


def apply_options(c, args):
    """The bench's variant switches on context c."""
    for flag, name in ((args.deterministic, "deterministic"), (args.bwd_per_splat, "bwd_per_splat")):
        if flag:
            c.set_option(name, True)
    if args.no_split:
        c.set_option("split", False)
    if args.split_forward:
        c.set_option("split_forward", True)


def bench_config(wl, args, pairs, world):
    """The `config` object of the JSON line; both arms print the same one."""
    return {"workload": workload_label(wl), "splats": wl.n, "width": wl.width, "height": wl.height,
            "pairs": int(pairs), "l2": "flushed between timed steps (256 MB write)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "backward_accumulation": "fixed point (deterministic)" if args.deterministic else "double atomics",
            "backward_loop_nest": "per splat (diagonal)" if args.bwd_per_splat else "per pixel",
            "long_lists": long_lists_label(args),
            "binning": "reserved arena (1.5 x the pair count), no host read-back" if args.reserved
            else "pair count read back every call",
            "e2e_binning": "reserved arena (1.5 x the pair count), no host read-back"}


def reference_arm(args):
    """The oracle, as it stands, on the host cores: every step is one whole
    frame (binning, forward, backward) cut into one tile-row band per core,
    the bands in parallel worker processes; the step time is the wall time."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor

    import oracle
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wl = gen.make(args.config)
    pairs = oracle.count_pairs(wl.splats, wl.depths, wl.width, wl.height)
    cores = len(os.sched_getaffinity(0))
    steps_ms = []
    with ProcessPoolExecutor(cores, mp_context=mp.get_context("spawn")) as pool:
        def one():
            t0 = time.perf_counter()
            list(pool.map(_oracle_band, [(args.config, k, cores) for k in range(cores)]))
            return (time.perf_counter() - t0) * 1e3
        for _ in range(args.warmup):
            one()
        for _ in range(args.steps):
            steps_ms.append(one())
    value = float(np.mean(steps_ms))
    line = {"metric": METRIC, "value": value, "unit": "ms/iter", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": value,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "impl": "reference",
            "config": bench_config(wl, args, pairs, 1),
            "cpu_baseline": {"value": value, "unit": "ms/iter", "cores": cores, "kind": "oracle",
                             "sample": f"every step the whole frame as {cores} tile-row bands (each bins "
                                       "every splat against its rows, then forward and backward), one "
                                       "worker process per band, wall time"},
            "e2e": {"value": value, "unit": "ms/iter", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def roofline_for(kind, counters, pairs, wl, ms, peaks, alu):
    """Algorithmic work of one launch against the measured FP32 / SFU / HBM peaks."""
    ops = FWD_OPS if kind == "forward" else BWD_OPS
    fp32 = sum(ops[k] * counters[k] for k in ops)
    sfu = counters["n_exp"] + (counters["n_contrib"] if kind == "backward" else 0)
    px = wl.width * wl.height
    if kind == "forward":
        bytes_ = pairs * (36 + 4) + px * 24
    else:
        bytes_ = pairs * (36 + 4) + px * (16 + 4 + 4) + wl.n * 36 * 2
    fp32_peak = alu["fp32_lane_ops_per_s"]
    sfu_peak = alu["sfu_lane_ops_per_s"]
    hbm_peak = peaks["hbm_gbs"] * 1e9
    t = {"alu": fp32 / fp32_peak, "sfu": sfu / sfu_peak, "hbm": bytes_ / hbm_peak}
    bound = max(t, key=t.get)
    sec = ms * 1e-3
    if bound == "hbm":
        achieved, peak, unit = bytes_ / sec / 1e9, peaks["hbm_gbs"], "GB/s"
    elif bound == "alu":
        achieved, peak, unit = fp32 / sec / 1e9, fp32_peak / 1e9, "Gop/s (fp32 lane ops)"
    else:
        achieved, peak, unit = sfu / sec / 1e9, sfu_peak / 1e9, "Gop/s (sfu lane ops)"
    formula = alu["formula_fp32_lane_ops_per_s"] if bound == "alu" else alu["formula_sfu_lane_ops_per_s"]
    return {"kernel": kind, "bound": "alu" if bound in ("alu", "sfu") else "hbm",
            "pipe": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": ncu_traffic(kind, wl.name),
            "peak_source": ("measured HBM copy (MEASURED_PEAKS.json)" if bound == "hbm" else
                            f"measured: the {'FFMA' if bound == 'alu' else 'ex2'} rate kernel (gsr_peak_kernel) "
                            f"timed in this run, {alu['sms']} SMs"),
            "peak_formula": None if bound == "hbm" else formula / 1e9,
            "algorithmic": {"fp32_ops": fp32, "sfu_ops": sfu, "bytes": bytes_}}


def measure_alu_peaks(gsr, ctx, dev, stream, reps=5):
    """FP32 (FFMA) and SFU (ex2) lane-operation rates of this GPU, from the
    library's rate kernels timed with CUDA events (best of `reps` launches of
    about 2 ms each after warm-up), beside the formula SMs x lanes x max clock."""
    import torch
    sink = torch.zeros(1, dtype=torch.float32, device=dev)
    props = torch.cuda.get_device_properties(dev)
    sms = int(props.multi_processor_count)
    out = {"sms": sms}
    for kind, iters in (("ffma", 16384), ("ex2", 2048)):
        rates = []
        for r in range(3 + reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ops = gsr.peak_kernel(ctx, kind, iters, sink, stream=stream)
            b.record(stream)
            b.synchronize()
            if r >= 3:
                rates.append(ops / (a.elapsed_time(b) * 1e-3))
        out["fp32_lane_ops_per_s" if kind == "ffma" else "sfu_lane_ops_per_s"] = float(max(rates))
    mhz = measured_peaks()["sm_max_mhz"]
    out["formula_fp32_lane_ops_per_s"] = sms * FP32_LANES_PER_SM * mhz * 1e6
    out["formula_sfu_lane_ops_per_s"] = sms * SFU_LANES_PER_SM * mhz * 1e6
    out["formula"] = f"{sms} SMs x {FP32_LANES_PER_SM} FP32 / {SFU_LANES_PER_SM} SFU lanes x {mhz:.0f} MHz"
    return out


# Algorithmic bytes per Gaussian of the projection kernels: the forward reads a
# 56-byte Gaussian and writes a 36-byte Splat2D and a 4-byte depth; the
# backward reads the Gaussian and its 36-byte Splat2D gradient and writes a
# 56-byte gradient.
PROJ_BYTES = {"project_forward": 56 + 36 + 4, "project_backward": 56 + 36 + 56}


def time_projection(gsr, ctx, dev, stream, flush, steps, warmup, peaks):
    """Times the projection forward and backward on the Lego-shaped 3-D scene
    (409,660 Gaussians, one 800x800 view), each launch alone between L2 flushes."""
    import torch

    sc = gen.lego_scene()
    g = torch.from_numpy(sc.gaussians).to(dev)
    G = torch.from_numpy(sc.dl_dsplat).to(dev)
    sp = torch.empty((sc.n, 9), dtype=torch.float32, device=dev)
    d = torch.empty((sc.n,), dtype=torch.float32, device=dev)
    dg = torch.empty((sc.n, 14), dtype=torch.float32, device=dev)
    calls = {"project_forward": lambda: gsr.project_forward(ctx, g, sc.camera, sp, d),
             "project_backward": lambda: gsr.project_backward(ctx, g, sc.camera, G, dg)}
    out = {"workload": f"lego_scene: {sc.n:,} Gaussians, 800x800 view, seed 3", "gaussians": sc.n}
    for name, call in calls.items():
        for i in range(warmup):
            flush.fill_(float(i))
            call()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            flush.fill_(float(i))
            evs[i][0].record(stream)
            call()
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        ms = np.array([a.elapsed_time(b) for a, b in evs])
        gbs = PROJ_BYTES[name] * sc.n / (float(ms.mean()) * 1e-3) / 1e9
        out[name] = {"ms": float(ms.mean()), "ms_median": float(np.median(ms)),
                     "bytes_per_gaussian": PROJ_BYTES[name],
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"],
                                  "traffic": ncu_traffic(name, "lego_scene")}}
    return out


def time_graph(gsr, ctx, wl, sp, dp, dl, out, fT, last, grad, dev, stream, flush, steps):
    """The whole step (binning with a reservation, forward, backward) replayed
    from one captured CUDA graph, against the same step with direct calls on
    the same context, alternating, between L2 flushes; medians.  ctx must have
    a reservation (a graph cannot hold the default binning's read-back)."""
    import torch

    def direct():
        b = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
        gsr.rasterize_forward(ctx, sp, b, out, fT, last)
        gsr.rasterize_backward(ctx, sp, b, dl, fT, last, grad)

    direct()
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            direct()
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)

    def run(graph):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            flush.fill_(float(i))
            evs[i][0].record(stream)
            if graph:
                g.replay()
            else:
                direct()
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return float(np.median([a.elapsed_time(b) for a, b in evs]))

    res = {"direct_ms": [], "graph_ms": []}
    for _ in range(3):
        res["direct_ms"].append(run(False))
        res["graph_ms"].append(run(True))
    return {"direct_ms": float(np.median(res["direct_ms"])), "graph_ms": float(np.median(res["graph_ms"])),
            "note": "binning, forward and backward as one graph replay against direct calls; medians of 3 x "
                    f"{steps} steps"}


# Frames timed beside the headline one (same step, same L2 flush): the pages'
# pair density, and a close-up whose crowded tiles the split serves, with and
# without the forward's split.
OTHER_CONFIGS = (("lego_pages", {}), ("lego_far", {}), ("lego_far", {"split_forward": True}))


def time_other_config(gsr, name, options, args, dev, stream, flush, steps, warmup):
    import torch
    wl = gen.make(name)
    ctx = gsr.Context(dev.index or 0)
    apply_options(ctx, args)
    for opt, value in options.items():
        ctx.set_option(opt, value)
    sp, dp, dl = (torch.from_numpy(a).to(dev) for a in (wl.splats, wl.depths, wl.dl_dout))
    npx = wl.width * wl.height
    out = torch.empty((npx, 4), dtype=torch.float32, device=dev)
    fT = torch.empty((npx,), dtype=torch.float32, device=dev)
    last = torch.empty((npx,), dtype=torch.int32, device=dev)
    grad = torch.empty((wl.n, 9), dtype=torch.float32, device=dev)

    def step(evs):
        evs[0].record(stream)
        bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
        evs[1].record(stream)
        gsr.rasterize_forward(ctx, sp, bins, out, fT, last)
        evs[2].record(stream)
        gsr.rasterize_backward(ctx, sp, bins, dl, fT, last, grad)
        evs[3].record(stream)

    for k in range(warmup):
        flush.fill_(float(k))
        step([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        flush.fill_(float(i))
        step(evs[i])
    torch.cuda.synchronize(dev)
    t = np.array([[e[k].elapsed_time(e[k + 1]) for k in range(3)] + [e[0].elapsed_time(e[3])] for e in evs])
    pairs = ctx.num_pairs()
    ctx.close()
    return {"workload": workload_label(wl), "options": options, "splats": wl.n, "pairs": int(pairs),
            "pairs_per_splat": pairs / wl.n, "steps": steps, "ms_per_step": float(t[:, 3].mean()),
            "stages_ms": {"bin": float(t[:, 0].mean()), "forward": float(t[:, 1].mean()),
                          "backward": float(t[:, 2].mean())}}


def gpu_arm(args):
    import torch

    import gaussian_splatting_tile_bin_gb300 as gsr

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = gen.make(args.config)
    ctx = gsr.Context(local)
    apply_options(ctx, args)
    stream = torch.cuda.current_stream(dev)

    sp = torch.from_numpy(wl.splats).to(dev)
    dp = torch.from_numpy(wl.depths).to(dev)
    dl = torch.from_numpy(wl.dl_dout).to(dev)
    npx = wl.width * wl.height
    out = torch.empty((npx, 4), dtype=torch.float32, device=dev)
    fT = torch.empty((npx,), dtype=torch.float32, device=dev)
    last = torch.empty((npx,), dtype=torch.int32, device=dev)
    grad = torch.empty((wl.n, 9), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    # One binning that reads its count back sizes the reservations (setup,
    # outside any timing) of the contexts that read nothing back: the e2e
    # contexts, the graph's, and the timed one with --reserved.
    reserve = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height).num_pairs * 3 // 2
    if args.reserved:
        ctx.reserve_pairs(reserve)

    def step(evs):
        evs[0].record(stream)
        bins = gsr.bin_splats(ctx, sp, dp, wl.width, wl.height)
        evs[1].record(stream)
        gsr.rasterize_forward(ctx, sp, bins, out, fT, last)
        evs[2].record(stream)
        gsr.rasterize_backward(ctx, sp, bins, dl, fT, last, grad)
        evs[3].record(stream)
        return bins

    def new_events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    sampler = ClockSampler(local)
    sampler.start()
    # Warm-up: W steps, then more untimed steps until ~1.5 s has passed so the
    # clock sampler sees the GPU under this load before the timed region.
    t_warm = time.perf_counter()
    k = 0
    while k < args.warmup or time.perf_counter() - t_warm < args.min_warm_s:
        flush.fill_(float(k))
        step(new_events())
        k += 1
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)

    launches0 = ctx.launch_count()
    evs = [new_events() for _ in range(args.steps)]
    wall0 = time.perf_counter()
    pairs = 0
    for i in range(args.steps):
        flush.fill_(float(i))      # L2 flush between timed steps (outside the events)
        step(evs[i])
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    launches = ctx.launch_count() - launches0
    pairs = ctx.num_pairs()          # raises if a step exceeded the reservation
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)

    bin_ms = np.array([e[0].elapsed_time(e[1]) for e in evs])
    fwd_ms = np.array([e[1].elapsed_time(e[2]) for e in evs])
    bwd_ms = np.array([e[2].elapsed_time(e[3]) for e in evs])
    tot_ms = np.array([e[0].elapsed_time(e[3]) for e in evs])

    # e2e: every step uploads its inputs from pinned host memory and reads its
    # gradients and image back.  Steps alternate between two contexts (each its
    # own arena) on two streams, so one step's copies overlap the other's
    # kernels; the time is the wall time of the whole sequence on the device.
    e2e = None
    if not args.no_e2e:
        h_sp = torch.from_numpy(wl.splats).pin_memory()
        h_dp = torch.from_numpy(wl.depths).pin_memory()
        h_dl = torch.from_numpy(wl.dl_dout).pin_memory()
        slots = []
        for k in range(2):
            c2 = gsr.Context(local)
            c2.reserve_pairs(reserve)
            apply_options(c2, args)
            slots.append({
                "ctx": c2, "stream": torch.cuda.Stream(dev),
                "sp": torch.empty_like(sp), "dp": torch.empty_like(dp), "dl": torch.empty_like(dl),
                "out": torch.empty_like(out), "fT": torch.empty_like(fT), "last": torch.empty_like(last),
                "grad": torch.empty_like(grad),
                "h_grad": torch.empty((wl.n, 9), dtype=torch.float32).pin_memory(),
                "h_out": torch.empty((npx, 4), dtype=torch.float32).pin_memory()})

        def e2e_step(i):
            sl = slots[i % 2]
            with torch.cuda.stream(sl["stream"]):
                sl["sp"].copy_(h_sp, non_blocking=True)
                sl["dp"].copy_(h_dp, non_blocking=True)
                sl["dl"].copy_(h_dl, non_blocking=True)
                b = gsr.bin_splats(sl["ctx"], sl["sp"], sl["dp"], wl.width, wl.height)
                gsr.rasterize_forward(sl["ctx"], sl["sp"], b, sl["out"], sl["fT"], sl["last"])
                gsr.rasterize_backward(sl["ctx"], sl["sp"], b, sl["dl"], sl["fT"], sl["last"], sl["grad"])
                sl["h_grad"].copy_(sl["grad"], non_blocking=True)
                sl["h_out"].copy_(sl["out"], non_blocking=True)

        def e2e_run(nsteps):
            torch.cuda.synchronize(dev)
            begin, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            begin.record(stream)
            for sl in slots:
                sl["stream"].wait_event(begin)
            for i in range(nsteps):
                e2e_step(i)
            for sl in slots:
                ev = torch.cuda.Event()
                ev.record(sl["stream"])
                stream.wait_event(ev)
            end.record(stream)
            end.synchronize()
            return begin.elapsed_time(end)

        def e2e_run_threads(nsteps):
            # One host thread per context: one context's binning waits for its
            # stream (the pair count) while the other thread keeps queueing.
            import threading
            torch.cuda.synchronize(dev)
            begin, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            begin.record(stream)
            for sl in slots:
                sl["stream"].wait_event(begin)
            errors = []

            def worker(k):
                try:
                    torch.cuda.set_device(dev)
                    for i in range(k, nsteps, 2):
                        e2e_step(i)
                except Exception as e:  # surfaced below
                    errors.append(e)

            threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
            for t in threads:
                t.start()
            for t in threads:
                t.join()
            if errors:
                raise errors[0]
            for sl in slots:
                ev = torch.cuda.Event()
                ev.record(sl["stream"])
                stream.wait_event(ev)
            end.record(stream)
            end.synchronize()
            return begin.elapsed_time(end)

        e2e_run(max(4, args.warmup))
        e2e_one_ms = e2e_run(args.steps)
        e2e_run_threads(max(4, args.warmup))
        e2e_two_ms = e2e_run_threads(args.steps)
        e2e_total_ms = min(e2e_one_ms, e2e_two_ms)
        # The copies brought back the same results as the device-resident steps
        # (the gradients up to the order of their double-precision sums).
        if not torch.equal(slots[0]["h_out"], out.cpu()) or not torch.allclose(
                slots[0]["h_grad"], grad.cpu(), rtol=1e-6, atol=1e-9):
            raise RuntimeError("e2e results differ from the device-resident run")
        h2d = (wl.splats.nbytes + wl.depths.nbytes + wl.dl_dout.nbytes)
        d2h = wl.n * 9 * 4 + npx * 16
        e2e_val = job_ms_per_iter(e2e_total_ms, args.steps, world, dev)
        e2e = {"value": e2e_val, "unit": "ms/iter", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "pipelining": "two contexts on two streams; a step's copies overlap the other's kernels; "
                             "the faster of one host thread alternating the contexts and one thread per context",
               "one_thread_ms_per_iter": e2e_one_ms / args.steps,
               "two_threads_ms_per_iter": e2e_two_ms / args.steps}

    graph = None
    if args.graph:
        gctx = gsr.Context(local)
        gctx.reserve_pairs(reserve)
        apply_options(gctx, args)
        graph = time_graph(gsr, gctx, wl, sp, dp, dl, out, fT, last, grad, dev, stream, flush, max(args.steps, 20))
        gctx.close()
    others = None
    if not args.no_other_configs and args.config == "lego_final" and world == 1:
        others = {name + "".join("+" + k for k in opts): time_other_config(
                      gsr, name, opts, args, dev, stream, flush, max(args.steps, 20), max(args.warmup, 3))
                  for name, opts in OTHER_CONFIGS}
    peaks = measured_peaks()
    # Binning against HBM: N·40 B of splats and depths read, each pair's 12-byte
    # key and index written once and read and written by every executed pair
    # pass, 8 B per pair for the range extraction, 8 B per tile of ranges.  The
    # pair arrays (12 B x pairs) stay in L2 at this size, so the kernels run
    # against L2 rather than HBM bandwidth.
    st = ctx.bin_stats()
    k_pass = bin(st["tile_pass_mask"]).count("1")
    bin_bytes = wl.n * 40 + pairs * 12 * (1 + 2 * k_pass) + pairs * 8 + \
        ((wl.width + 15) // 16) * ((wl.height + 15) // 16) * 8
    bin_gbs = bin_bytes / (float(bin_ms.mean()) * 1e-3) / 1e9
    roofline_bin = {"kernel": "bin (all binning launches)", "bound": "hbm", "achieved": bin_gbs,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": bin_gbs / peaks["hbm_gbs"],
                    "algorithmic_bytes": int(bin_bytes), "pair_passes": k_pass,
                    "radix_passes": st["radix_passes"],
                    "note": "pair arrays are L2-resident at this size"}
    projection = None
    if not args.no_projection:
        projection = time_projection(gsr, ctx, dev, stream, flush, max(args.steps, 20), max(args.warmup, 3),
                                     peaks)

    alu = None if args.no_alu_peaks else measure_alu_peaks(gsr, ctx, dev, stream)
    rows = sampler.stop()
    clocks = ClockSampler.summarize(rows)

    value = job_ms_per_iter(float(tot_ms.sum()), args.steps, world, dev)

    line = {"metric": METRIC, "value": value, "unit": "ms/iter", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": float(tot_ms.mean()),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": bench_config(wl, args, pairs, world),
            "ms_per_step_median": float(np.median(tot_ms)), "ms_per_step_std": float(np.std(tot_ms)),
            "stages_ms": {"bin": float(bin_ms.mean()), "forward": float(fwd_ms.mean()),
                          "backward": float(bwd_ms.mean()),
                          "bin_median": float(np.median(bin_ms)),
                          "forward_median": float(np.median(fwd_ms)),
                          "backward_median": float(np.median(bwd_ms))},
            "wall_s": wall, "gpu_launches": int(launches), "clocks": clocks}
    if e2e:
        line["e2e"] = e2e
    if projection:
        line["projection"] = projection
    line["roofline_bin"] = roofline_bin
    line["alu_peaks"] = alu
    if graph:
        line["graph"] = graph
    if others:
        line["other_configs"] = others

    if rank == 0 and world == 1 and not args.no_cpu_baseline and alu:
        cb = cpu_baseline(wl)
        line["cpu_baseline"] = {"value": cb["ms"], "unit": "ms/iter", "cores": 1, "kind": "oracle",
                                "sample": "the whole workload once (binning, forward, backward), "
                                          "single thread",
                                "stages_ms": {"bin": cb["bin_ms"], "forward": cb["fwd_ms"],
                                              "backward": cb["bwd_ms"]}}
        if not args.no_cpu_all_cores:
            ms_all, cores = cpu_baseline_all_cores(args.config)
            line["cpu_baseline_all_cores"] = {
                "value": ms_all, "unit": "ms/iter", "cores": cores, "kind": "oracle",
                "sample": f"the whole frame as {cores} tile-row bands (each bins every splat against "
                          "its rows, then forward and backward), one worker process per band, wall time"}
        rf = roofline_for("forward", cb["fwd_counters"], cb["pairs"], wl, float(fwd_ms.mean()), peaks, alu)
        rb = roofline_for("backward", cb["bwd_counters"], cb["pairs"], wl, float(bwd_ms.mean()), peaks, alu)
        dom = rb if bwd_ms.mean() >= fwd_ms.mean() else rf
        line["roofline"] = dom
        line["roofline_other"] = rf if dom is rb else rb
        line["counters"] = {"forward": cb["fwd_counters"], "backward": cb["bwd_counters"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return reference_arm(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
