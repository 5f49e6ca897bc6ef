#!/usr/bin/env python3
"""Benchmark of the GB300 pillar voxelizer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload kitti|dense|adversarial|tiny|uniform_<n>]

One step = one voxelization of one synthetic frame (the whole hot path: bin,
group, rank, emit, zero-fill) through the C ABI.  The default workload is the
KITTI-shaped 122,880-return frame (432 x 496 grid, 32 points per pillar,
16,000 pillars).  Inputs are resident in HBM before timing starts; the frame
buffers (input + all outputs) rotate over a set larger than twice the L2, so
every step reads and writes memory that is not in L2.  Times come from CUDA
events on the launching stream; with torchrun (N > 1) every rank voxelizes
its own frames (replicas, no collective on the data path) and the maximum
time over ranks is reported.

--impl reference times the CPU oracle (single-threaded C++) on the host on
the same workload, one frame per step.

Prints ONE JSON line (rank 0).
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
sys.path.insert(0, ROOT)

METRIC = "Mpoints/s voxelized per frame; achieved HBM GB/s vs GB300 peak"
SPIN_CYCLES = 2_000_000  # about 1 ms of GPU spin queued before each timed region
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="kitti")
    ap.add_argument("--order", default="canonical", choices=["canonical", "unordered"],
                    help="canonical order (default) or the page's own unordered contract")
    ap.add_argument("--op", default="voxelize", choices=["voxelize", "downsample", "fps"],
                    help="voxelize (PointPillars tensors), voxel-grid centroid downsampling, or farthest point "
                         "sampling (workload lidar65k)")
    ap.add_argument("--no-graph", action="store_true",
                    help="time plain stream launches instead of one CUDA graph holding the K timed launches")
    ap.add_argument("--batch", type=int, default=1,
                    help="frames per launch (pv_voxelize_batch when > 1; different frames of the workload)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU oracle sample length")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def max_over_ranks(value, device=None):
    """Maximum of a per-rank float over the process group (identity at N = 1)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(points_per_frame, steps, world, region_ms):
    """Mpoints/s over all ranks: every rank voxelizes `steps` frames of its own."""
    return world * points_per_frame * steps / (region_ms * 1e-3) / 1e6


def algorithmic_bytes(n, max_points, max_voxels):
    # Input read once (16 B/point) + every output byte written once:
    # voxels 16*K B, coords 12 B, counts 4 B per pillar row, plus V (4 B).
    return 16 * n + max_voxels * (16 * max_points + 16) + 4


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


HOST_SIDE_MARKER = b"// ------------------------------------------------------------ host side"

# The source files of each profiled kernel: the shared device header and the
# kernel's own file (farthest point sampling is one file).
KERNEL_SOURCES = {
    "pv_voxelize_kernel": ("pv_device.cuh", "pv_ordered.cu"),
    "pv_unordered_kernel": ("pv_device.cuh", "pv_unordered.cu"),
    "pv_downsample_kernel": ("pv_device.cuh", "pv_downsample.cu"),
    "pv_fps_kernel": ("pv_fps.cu",),
}


def kernel_sha(kernel="pv_voxelize_kernel"):
    """SHA-256 of the device code of the files that hold the kernel: each
    file up to its host-side marker (launch, planning and ABI code after it
    can change without changing what a profile measured), with line
    comments, trailing blanks and empty lines left out (comment edits do not
    change the kernel either)."""
    code = []
    for name in KERNEL_SOURCES[kernel]:
        src = os.path.join(ROOT, "lidar_point_cloud_gb300", "csrc", name)
        with open(src, "rb") as f:
            text = f.read()
        cut = text.find(HOST_SIDE_MARKER)
        for line in (text[:cut] if cut >= 0 else text).split(b"\n"):
            line = line.split(b"//", 1)[0].rstrip()
            if line:
                code.append(line)
    return hashlib.sha256(b"\n".join(code)).hexdigest()


def profiled_traffic(workload, kernel="pv_voxelize_kernel"):
    """DRAM bytes per launch from the committed ncu summary, if it still
    describes the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != kernel_sha(kernel):
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile

        fd, self.path = tempfile.mkstemp(prefix="pv_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        os.unlink(self.path)
        busy = [r for r in rows if r[4].isdigit() and int(r[4]) > 0] or rows
        sm = [float(r[1]) for r in busy if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in busy if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(busy)}


def oracle_op(P, op="voxelize"):
    """The oracle pass a workload takes: the 3-D pass when the grid has layers."""
    import oracle

    if op == "downsample":
        return "downsample"
    return "voxelize3d" if oracle.grid3d(P.point_cloud_range, P.voxel_size)[1][2] > 1 else "voxelize"


def host_cpu():
    """The host's CPU model and logical core count."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return {"model": model or "unknown", "nproc": os.cpu_count()}


class OneCore:
    """Pins the calling process to one core (the last it may run on) and
    restores its affinity afterwards."""

    def __enter__(self):
        self.prev = os.sched_getaffinity(0)
        self.core = max(self.prev)
        os.sched_setaffinity(0, {self.core})
        return self

    def __exit__(self, *exc):
        os.sched_setaffinity(0, self.prev)


def oracle_runs(pts, P, op, reps):
    """Per-run durations (s) of the oracle pass on one frame, measured with
    steady_clock inside the C++ library (no Python in the timed region)."""
    import oracle

    return oracle.time_passes(oracle_op(P, op), pts, P.point_cloud_range, P.voxel_size, P.max_points,
                              P.max_voxels, reps) * 1e-9


def cpu_baseline(pts, P, seconds, op="voxelize", what="the full frame"):
    """The single-threaded C++ oracle on one host core: the median of at least
    five runs (three for frames over a second), about `seconds` of work in all."""
    n = pts.shape[0]
    with OneCore() as pin:
        first = float(oracle_runs(pts, P, op, 1)[0])
        reps = int(max(3 if first > 1.0 else 5, min(1000, seconds / max(first, 1e-6))))
        runs = oracle_runs(pts, P, op, reps)
    med = float(statistics.median(runs))
    return {"value": round(n / med / 1e6, 3), "unit": "Mpoints/s", "cores": 1, "kind": "oracle",
            "median_ms": round(med * 1e3, 3), "runs": int(reps), "pinned_core": pin.core, "host": host_cpu(),
            "sample": f"{reps} runs on {what} ({sum(runs):.1f} s), median per run on steady_clock inside the "
                      f"single-threaded C++ oracle ({oracle_op(P, op)}), process pinned to one core"}


def run_reference(args, rank, world):
    import numpy as np

    from lidar_point_cloud_gb300 import synth

    if rank != 0:
        return
    import oracle

    lib = oracle.load()
    if args.op == "fps":
        B = max(1, args.batch)
        clouds = [synth.fps_cloud(1 + b) for b in range(B)]
        M = synth.FPS_SAMPLES
        # A step is a bounded sample: the first S samples of each cloud (the
        # cost is linear in the samples), S sized so that the warm-up and the
        # timed steps take about a minute; the rate counts S/M of a cloud.
        t0 = time.perf_counter()
        oracle.fps(clouds[0], 64, 0, lib)
        per_sample = (time.perf_counter() - t0) / 64
        S = int(max(16, min(M, 60.0 / max(1, args.steps + args.warmup) / (B * per_sample))))
        for _ in range(args.warmup):  # untimed, as on the GPU arm
            for c in clouds:
                oracle.fps(c, S, 0, lib)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            for c in clouds:
                oracle.fps(c, S, 0, lib)
        el = time.perf_counter() - t0
        value = synth.FPS_POINTS * B * args.steps * (S / M) / el / 1e6
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "Mpoints/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 * el / args.steps * (M / S), 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": f"lidar65k: {synth.WORKLOADS['lidar65k']}", "op": "fps", "clouds_per_launch": B},
                "cpu_baseline": {"value": round(value, 3), "unit": "Mpoints/s", "cores": 1, "kind": "oracle",
                                 "sample": f"the first {S} of {M} samples of {B} cloud(s) per step ({args.steps} steps; "
                                           f"rate scaled by {M}/{S}, the cost being linear in the samples), C++ O(N*M) loop"},
                "e2e": {"value": round(value, 3), "unit": "Mpoints/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    if args.batch > 1:
        pts, frame_off, P = synth.make_batch(args.workload, args.batch)
        frames = [pts[frame_off[b]:frame_off[b + 1]] for b in range(args.batch)]
    else:
        pts, P = synth.make(args.workload)
        frames = [pts]

    # A step is one oracle pass per frame, timed on steady_clock inside the
    # C++ library with the process pinned to one core; a bounded sample: when
    # whole frames would make the warm-up and timed steps run past about a
    # minute, each step takes the first points of each frame instead (the
    # metric counts the points done).
    with OneCore() as pin:
        t_full = sum(float(oracle_runs(f, P, args.op, 1)[0]) for f in frames)
        runs = max(1, args.steps + args.warmup)
        if runs * t_full > 60.0:
            keep = max(4096 / max(1, max(f.shape[0] for f in frames)), 60.0 / (runs * t_full))
            frames = [f[:max(1, int(f.shape[0] * keep))] for f in frames]
        per_frame = [oracle_runs(f, P, args.op, args.warmup + args.steps)[args.warmup:] for f in frames]
    el = float(sum(np.sum(t) for t in per_frame))
    n = sum(f.shape[0] for f in frames)
    value = n * args.steps / el / 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "Mpoints/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * el / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": (f"{args.workload} x{args.batch} frames per launch: " if args.batch > 1 else
                                f"{args.workload}: ") + synth.WORKLOADS[args.workload], "N": n,
                   "max_points": P.max_points, "max_voxels": P.max_voxels, "frames_per_launch": args.batch},
        "cpu_baseline": {"value": round(value, 3), "unit": "Mpoints/s", "cores": 1, "kind": "oracle",
                         "pinned_core": pin.core, "host": host_cpu(),
                         "sample": (f"{args.batch} frame(s) per step, {n:,} of {pts.shape[0]:,} points "
                                    f"({'whole frames' if n == pts.shape[0] else 'the first points of each frame'}), "
                                    f"{args.steps} steps, each pass on steady_clock inside the single-threaded C++ "
                                    "std::map oracle, process pinned to one core")},
        "e2e": {"value": round(value, 3), "unit": "Mpoints/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# Plain fp32 lanes of the GPU (no multiply-add is used by the FPS distances):
# 152 SMs x 128 lanes x 2.07 GHz maximum SM clock.
FP32_LANES_PER_SM = 128


def run_fps(args, rank, world, local_rank):
    """Farthest point sampling: B clouds of 65,536 points, 4,096 samples each."""
    import numpy as np
    import torch

    import lidar_point_cloud_gb300 as pv
    from lidar_point_cloud_gb300 import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    B, N, M = max(1, args.batch), synth.FPS_POINTS, synth.FPS_SAMPLES
    clouds = np.stack([synth.fps_cloud(1 + b) for b in range(B)])
    src = torch.from_numpy(clouds).to(dev)
    pts = src if B > 1 else src[0]
    lead = (B,) if B > 1 else ()
    idx = torch.empty(lead + (M,), dtype=torch.int32, device=dev)
    smp = torch.empty(lead + (M, 4), dtype=torch.float32, device=dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        pv.fps_into(pts, M, idx, smp, status, 0, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError("device status")
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize(dev)
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for k in range(args.steps):
        starts[k].record(stream)
        step()
        ends[k].record(stream)
    r1.record(stream)
    torch.cuda.synchronize(dev)
    region_ms = max_over_ranks(r0.elapsed_time(r1), device=dev)
    kernel_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    t_soak = time.perf_counter()
    while sampler and time.perf_counter() - t_soak < 1.5:
        step()
        torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None
    if rank != 0:
        return
    value = whole_job_rate(B * N, args.steps, world, region_ms)
    ops = 8.0 * N * (M - 1) * B  # 3 subtractions, 3 products, 2 sums per point per sample
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak_ops = sms * FP32_LANES_PER_SM * 2.07e9
    achieved = ops / (kernel_ms * 1e-3)
    # End to end: pinned host clouds in, indices and samples out.
    pin = torch.from_numpy(clouds).pin_memory()
    pin_in = pin if B > 1 else pin[0]
    h_idx = torch.empty(idx.shape, dtype=torch.int32).pin_memory()
    h_smp = torch.empty(smp.shape, dtype=torch.float32).pin_memory()
    e_steps = max(3, args.e2e_steps // 10)
    t0 = time.perf_counter()
    for _ in range(e_steps):
        d = pin_in.to(dev, non_blocking=True)
        pv.fps_into(d, M, idx, smp, status, 0, stream)
        h_idx.copy_(idx, non_blocking=True)
        h_smp.copy_(smp, non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_s = time.perf_counter() - t0
    cpu = None
    if not args.no_cpu_baseline:
        import oracle

        lib = oracle.load()
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds or reps == 0:
            oracle.fps(clouds[0], M, 0, lib)
            reps += 1
        el = time.perf_counter() - t0
        cpu = {"value": round(N * reps / el / 1e6, 3), "unit": "Mpoints/s", "cores": 1, "kind": "oracle",
               "sample": f"{reps} full sampling(s) of one cloud ({el:.1f} s), single-threaded C++ O(N*M) loop"}
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "Mpoints/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(region_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"lidar65k: {synth.WORKLOADS['lidar65k']}", "op": "fps", "clouds_per_launch": B,
                   "N": N, "samples": M, "launch": f"{B} cluster(s), one a cloud: 16 CTAs x 256 threads (16 points a thread in registers) while the clouds fit on the GPU at once, else 8 CTAs x 256 (32 points a thread)",
                   "l2": "the cloud is read once per launch into registers; no memory traffic between samples",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "alu", "achieved": round(achieved / 1e9, 1), "peak": round(peak_ops / 1e9, 1),
                     "unit": "Gop/s", "frac": round(achieved / peak_ops, 4),
                     "traffic": profiled_traffic("lidar65k" + (f"_x{B}" if B > 1 else ""), "pv_fps_kernel"),
                     "peak_source": f"derived: {sms} SMs x {FP32_LANES_PER_SM} fp32 lanes x 2.07 GHz",
                     "kernel": "pv_fps_kernel", "ops_per_launch": ops,
                     "avg_launch_us": round(kernel_ms * 1e3, 3)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(N * B * e_steps / e2e_s / 1e6, 3), "unit": "Mpoints/s",
                "h2d_bytes_per_step": 16 * N * B, "d2h_bytes_per_step": 4 * M * B + 16 * M * B,
                "api": "fps_into with pinned host copies in and out, synchronous", "steps": e_steps},
        "gpu_launches": args.steps, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def run_gb300(args, rank, world, local_rank):
    import numpy as np
    import torch

    import lidar_point_cloud_gb300 as pv
    from lidar_point_cloud_gb300 import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    Bf = args.batch
    if Bf > 1:
        pts, frame_off, P = synth.make_batch(args.workload, Bf)
    else:
        pts, P = synth.make(args.workload)
        frame_off = [0, pts.shape[0]]
    n, K, M = pts.shape[0], P.max_points, P.max_voxels
    ds = args.op == "downsample"
    if ds and (Bf > 1 or args.order != "canonical"):
        raise SystemExit("--op downsample takes one frame per launch in the canonical order")
    plan = pv.query_plan(n, P.point_cloud_range, P.voxel_size, K, M)
    if ds:  # input once; centroid (16 B), coordinates (12 B) and count (4 B) of every row, V
        bytes_launch = 16 * n + M * 32 + 4
    else:   # input once, every output byte of every frame once
        bytes_launch = 16 * n + Bf * (M * (16 * K + 16) + 4)
    frame_bytes = bytes_launch
    R = max(2, -(-2 * L2_BYTES // frame_bytes))
    src = torch.from_numpy(pts).to(dev)
    inputs = [src.clone() for _ in range(R)]
    outs = [(pv.alloc_downsample_outputs(M, dev) if ds else
             pv.alloc_batch_outputs(Bf, K, M, dev) if Bf > 1 else pv.alloc_outputs(K, M, dev)) for _ in range(R)]
    stream = torch.cuda.Stream(dev)  # a stream of its own (graph capture needs a non-default stream)
    torch.cuda.synchronize(dev)

    unordered = args.order == "unordered"
    if unordered and Bf > 1:
        raise SystemExit("--order unordered takes one frame per launch")
    kernel = "pv_downsample_kernel" if ds else "pv_unordered_kernel" if unordered else "pv_voxelize_kernel"

    def step(k):
        if ds:
            pv.downsample_into(inputs[k % R], P.point_cloud_range, P.voxel_size, M, outs[k % R], stream=stream)
        elif Bf > 1:
            pv.voxelize_batch_into(inputs[k % R], frame_off, P.point_cloud_range, P.voxel_size, K, M, outs[k % R],
                                   stream=stream)
        else:
            pv.voxelize_into(inputs[k % R], P.point_cloud_range, P.voxel_size, K, M, outs[k % R], stream=stream,
                             unordered=unordered)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize(dev)
    # Correctness guard on the last warm-up output (cheap: V only).
    v_dev = int(outs[(args.warmup - 1) % R][3].min().item()) if args.warmup else 0
    if v_dev < 0:
        raise RuntimeError(f"device status {v_dev}")

    dist = None
    if world > 1:
        import torch.distributed as dist

    use_graph = not args.no_graph
    graph = None
    if use_graph:
        # The K timed launches, captured once as one CUDA graph (the library's
        # calls are stream-ordered and allocate nothing once warm), so the
        # timed region holds exactly K launches without per-launch host work.
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for k in range(args.steps):
                step(args.warmup + k)
        with torch.cuda.stream(stream):
            graph.replay()  # untimed: first replay
        torch.cuda.synchronize(dev)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)

    def stream_launches():
        """K plain stream launches, an event pair around each."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(SPIN_CYCLES)  # the launches queue up behind it
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        for k in range(args.steps):
            starts[k].record(stream)
            step(args.warmup + k)
            ends[k].record(stream)
        r1.record(stream)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        return r0.elapsed_time(r1), [a.elapsed_time(b) for a, b in zip(starts, ends)]

    # Timed region: the K launches of the graph, replayed once; a spin kernel
    # queued first keeps the host's graph submission out of the region, so it
    # holds the K launches back to back whatever K is.
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if use_graph:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(SPIN_CYCLES)
        region0 = torch.cuda.Event(enable_timing=True)
        region1 = torch.cuda.Event(enable_timing=True)
        region0.record(stream)
        with torch.cuda.stream(stream):  # replay on the stream the events are recorded on
            graph.replay()
        region1.record(stream)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        region_ms = region0.elapsed_time(region1)
        # Launches back to back, no gaps to hide: the region over K.
        kernel_ms = [region_ms / args.steps]
        # The same K launches as plain stream launches, reported beside it.
        stream_region_ms, stream_ms = stream_launches()
    else:
        region_ms, kernel_ms = stream_launches()
        stream_region_ms, stream_ms = region_ms, kernel_ms
    # Keep the GPU busy (untimed) so the clock sampler sees at least ~1.5 s of load.
    t_soak = time.perf_counter()
    k = 0
    while sampler and time.perf_counter() - t_soak < 1.5:
        if use_graph:
            with torch.cuda.stream(stream):
                graph.replay()
            torch.cuda.synchronize(dev)
        else:
            step(k)
            k += 1
            if k % 256 == 0:
                torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop() if sampler else None

    region_ms = max_over_ranks(region_ms, device=dev)
    # Result check after timing: the last timed output against the first.
    last = outs[(args.warmup + args.steps - 1) % R]
    V = int(last[3].sum().item())

    if rank != 0:
        return
    value = whole_job_rate(n, args.steps, world, region_ms)
    avg_kernel_s = statistics.mean(kernel_ms) * 1e-3
    # Data-only bytes: the input once and the rows actually filled (V of them),
    # beside the padded contract's every output byte.
    if ds:
        data_bytes = 16 * n + V * 32 + 4
    else:
        data_bytes = 16 * n + V * (16 * K + 16) + 4 * Bf
    peak, peak_src = measured_peak()
    achieved = bytes_launch / avg_kernel_s / 1e9

    # End to end through the C ABI with host buffers (pinned), rank 0 only.
    pin_t = torch.from_numpy(pts).pin_memory()
    host_t = tuple(torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs[0])
    if ds:  # Python API: pinned host -> device, downsample_into, device -> pinned host

        def e2e_step():
            d_pts = pin_t.to(dev, non_blocking=True)
            pv.downsample_into(d_pts, P.point_cloud_range, P.voxel_size, M, outs[0], stream=stream)
            for h, d in zip(host_t, outs[0]):
                h.copy_(d, non_blocking=True)
            torch.cuda.synchronize(dev)
        api = "downsample_into with pinned host copies in and out, synchronous"
    elif Bf > 1:  # Python API: pinned host -> device, voxelize_batch_into, device -> pinned host

        def e2e_step():
            d_pts = pin_t.to(dev, non_blocking=True)
            pv.voxelize_batch_into(d_pts, frame_off, P.point_cloud_range, P.voxel_size, K, M, outs[0], stream=stream)
            for h, d in zip(host_t, outs[0]):
                h.copy_(d, non_blocking=True)
            torch.cuda.synchronize(dev)
        api = f"voxelize_batch_into ({Bf} frames) with pinned host copies in and out, synchronous"
    elif unordered:  # Python API: pinned host -> device, voxelize_into, device -> pinned host

        def e2e_step():
            d_pts = pin_t.to(dev, non_blocking=True)
            pv.voxelize_into(d_pts, P.point_cloud_range, P.voxel_size, K, M, outs[0], stream=stream, unordered=True)
            for h, d in zip(host_t, outs[0]):
                h.copy_(d, non_blocking=True)
            torch.cuda.synchronize(dev)
        api = "voxelize_into(unordered=True) with pinned host copies in and out, synchronous"
    else:
        def e2e_step():
            pv.voxelize_host(pin_t, P.point_cloud_range, P.voxel_size, K, M, out=host_t, stream=stream)
        api = ("voxelize_host -> pv_voxelize_host (C ABI, pinned host buffers read and written in place, synchronous; "
               "the result is the first V rows, each padded to max_points)")
    for _ in range(5):
        e2e_step()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        e2e_step()
    e2e_s = time.perf_counter() - t0
    d2h = sum(int(o.numel()) * 4 for o in outs[0])
    if api.startswith("voxelize_host"):  # rows [0, V) of voxels, coords and counts, and V
        d2h = int(host_t[3][0]) * (16 * K + 12 + 4) + 4
    e2e = {"value": round(n * args.e2e_steps / e2e_s / 1e6, 3), "unit": "Mpoints/s",
           "h2d_bytes_per_step": 16 * n, "d2h_bytes_per_step": d2h,
           "api": api, "steps": args.e2e_steps}

    cpu = None
    if not args.no_cpu_baseline:
        one = pts[:frame_off[1]] if Bf > 1 else pts
        cpu = cpu_baseline(one, P, args.cpu_seconds, args.op,
                           "the first frame" if Bf > 1 else "the full frame")

    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "Mpoints/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(region_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": (f"{args.workload} x{Bf} frames per launch: " if Bf > 1 else f"{args.workload}: ")
                        + synth.WORKLOADS[args.workload],
            "N": n, "V": V, "frames_per_launch": Bf, "grid": list(plan["grid"]), "max_points": K, "max_voxels": M,
            "table": (f"{plan['table_mode']}, {plan['table_slots']} slots" if Bf == 1 else
                      f"one key space per frame, {Bf} x {int(np.prod(plan['grid']))} voxel ids"),
            "launch": (f"1 cooperative kernel per step, {plan['ctas']} blocks x {plan['threads']} threads; "
                       + ("the K timed launches replayed as one CUDA graph; launch time = region / K" if use_graph
                          else "plain stream launches, one CUDA event pair per launch")),
            "l2": f"inputs+outputs rotate over {R} frame buffers ({R * frame_bytes / 2**20:.0f} MiB > 2x L2)",
            "parallelism": f"replicas x{world}",
            "order": args.order,
            "op": args.op,
        },
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(args.workload + (f"_x{Bf}" if Bf > 1 else ""), kernel),
            "peak_source": f"{peak_src} (hbm_gbs)", "kernel": kernel,
            "bytes_per_launch": bytes_launch, "avg_launch_us": round(avg_kernel_s * 1e6, 3),
            "median_launch_us": None if use_graph else round(statistics.median(kernel_ms) * 1e3, 3),
            "timing": {
                "graph_replay_us_per_launch": round(region_ms / args.steps * 1e3, 3) if use_graph else None,
                "stream_mean_us": round(statistics.mean(stream_ms) * 1e3, 3),
                "stream_median_us": round(statistics.median(stream_ms) * 1e3, 3),
                "stream_region_us_per_launch": round(stream_region_ms / args.steps * 1e3, 3),
                "note": "graph replay = K launches captured once, region over K; stream = the same K launches "
                        "issued one by one, an event pair around each; both regions start behind a spin kernel",
            },
            "data_bytes_per_launch": data_bytes,
            "frac_data": round(data_bytes / avg_kernel_s / 1e9 / peak, 4),
        },
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        if args.op == "fps":
            run_fps(args, rank, world, local_rank)
        else:
            run_gb300(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
