"""Benchmark of the sparse-weight direct convolution forward on GB300.

One step = one forward of one seeded synthetic layer (default: the 90 %
layer of the sparsity sweep, N=8, C=M=512, 28x28, 3x3, lognormal per-row
density -- the largest one-GPU layer in the 90-99 % range) through the C ABI
(spconv_forward), inputs resident in HBM.  The packing (spconv_pack) runs once
per weight set before timing, as in deployment, and is reported separately.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl ours|reference] [--no-layers]

Timing (default, --timing graph): W untimed warm-up steps, then the K steps
replayed back to back from CUDA graphs, each on its own copy of input,
weights and output, the copies together larger than twice the L2; CUDA events
on the launching stream around the region, a barrier and a device
synchronize on both sides, max over ranks.  --timing flush times each step
alone after a 256 MiB L2 flush instead.  Rank 0 prints one JSON line.

`layers`: every other seeded layer (ResNet-, VGG-, AlexNet-style, the rest of
the sweep) timed the same back-to-back way after the headline, each with its
µs/layer, roofline and in-core fractions and recorded DRAM traffic.

End to end (`e2e`): the headline layer through spconv_forward_host, one call
per step with the input and the result in page-locked host memory (the copies
to and from the GPU inside the timed events).

--impl reference times the CPU oracle (the only other implementation of this
path) on the host cores on the same layer; its `config` is the same dict.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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

import workloads  # noqa: E402
from sparse_weight_direct_gb300 import roofline  # noqa: E402

METRIC = "µs/layer and dense-equivalent TFLOP/s at 90–99% sparsity; % of roofline"
UNIT = "µs/layer"
FLUSH_BYTES = 256 << 20          # > 2x the 129 MB L2
SM_COUNT_NOMINAL = 152
FP32_LANES_PER_SM = 128
# Everything that decides what one launch of a kernel does: the kernel, its
# instances and the planner that picks the tiling (a plan change changes the
# traffic too).  One list per kernel, so a change to one leaves the other's
# recorded traffic valid.
_CSRC = os.path.join(ROOT, "sparse_weight_direct_gb300", "csrc")
KERNEL_SOURCES = {
    "spconv_fwd_kernel": [os.path.join(_CSRC, f) for f in (
        "spconv_kernel.cuh", "spconv_fwd.cu", "spconv_fwd_q1.cu", "spconv_fwd_q2.cu",
        "spconv_fwd_q4.cu", "spconv_fwd_q8.cu", "spconv_fwd_pairs.cu",
        "spconv_fwd_plane.cu", "spconv_fwd_cols.cu", "spconv_fwd_colpair.cu",
        "spconv_fwd_colpair5.cu", "spconv_fwd_tight.cu", "spconv_host.cpp",
        "spconv_internal.h")],
    "spconv_ws_kernel": [os.path.join(_CSRC, f) for f in (
        "spconv_kernel.cuh", "spconv_ws.cu", "spconv_host.cpp", "spconv_internal.h")],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0}, "fallback"


def fp32_peak_flops(sm_count: int, sm_mhz: float) -> float:
    """CUDA-core fp32 peak: SMs x 128 FMA lanes x 2 FLOP x clock."""
    return sm_count * FP32_LANES_PER_SM * 2.0 * sm_mhz * 1e6


def kernel_sha(kernel: str = "spconv_fwd_kernel") -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES[kernel]:
        with open(p, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def recorded_traffic(config: str, kernel: str = "spconv_fwd_kernel"):
    """DRAM bytes per launch from an ncu capture of this exact kernel source,
    or None (no capture, or the kernel changed since)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    sha = kernel_sha(kernel)
    with open(TRAFFIC_FILE) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == config \
                    and parts[1] == sha:
                return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(values, world: int, device=None):
    """Element-wise max of a list of floats over all ranks (the slowest rank
    sets the job's time).  Host plumbing only: one all_reduce of a few
    numbers, no data-path collective."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_us_per_layer(max_total_ms: float, steps: int, world: int) -> float:
    """Replicas: every rank runs `steps` layers in parallel, so the job
    processes steps * world layers in the slowest rank's time."""
    return max_total_ms * 1e3 / (steps * world)


def layer_numbers(L, nnz: int, entry_bytes: int = roofline.ENTRY_BYTES):
    E, F = L.E, L.F
    return {
        "useful_flop": roofline.useful_flops(nnz, L.N, E, F),
        "dense_flop": roofline.dense_equiv_flops(L.N, E, F, L.M, L.C, L.R, L.S),
        "alg_bytes": roofline.algorithmic_bytes(L.N, L.C, L.H, L.W, L.M, E, F, nnz, entry_bytes),
    }


def l2_method(timing: str) -> str:
    """How the timed steps keep L2 from serving their data (the same words on
    both arms of the benchmark, so their configs compare key for key)."""
    if timing == "flush":
        return "GPU: each timed step alone after a 256 MiB write that flushes L2"
    return ("GPU: inputs larger than L2 -- copies of input, weights and output, the steps "
            "replayed back to back from CUDA graphs")


def describe(L, fmt: str = "f32", timing: str = "graph"):
    """The workload a line's metric is measured on."""
    return {"workload": L.name, "N": L.N, "C": L.C, "H": L.H, "W": L.W, "M": L.M,
            "R": L.R, "S": L.S, "stride": L.stride, "pad": L.pad,
            "sparsity": round(1 - L.density, 4), "rows": L.rows,
            "weight_format": fmt, "l2": l2_method(timing)}


# --------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline leg)
# --------------------------------------------------------------------------

def time_oracle(L, rowptr, colidx, value, x, budget_s: float, steps: int = 1):
    """Time oracle.csr on a bounded sample of the layer: the first n images and
    first m output channels, sized so `steps` repeats fit in budget_s.
    Returns (us_per_layer, threads, sample_description, per-step seconds)."""
    import oracle
    # calibrate on one image and a slice of channels
    m_cal = max(1, min(L.M, 16))
    t0 = time.perf_counter()
    _, _, threads = oracle.csr(x[:1], rowptr[:m_cal + 1], colidx[:rowptr[m_cal]],
                               value[:rowptr[m_cal]], m_cal, L.R, L.S, L.stride, L.pad,
                               return_threads=True)
    t_cal = max(time.perf_counter() - t0, 1e-6)
    nnz_cal = max(int(rowptr[m_cal]), 1)
    per_nnz_img = t_cal / nnz_cal
    full = per_nnz_img * int(rowptr[-1]) * L.N
    target = max(budget_s / max(steps, 1), 1e-4)
    if full <= target:
        n_s, m_s = L.N, L.M
    else:
        n_s = max(1, min(L.N, int(target / (per_nnz_img * int(rowptr[-1])))))
        if n_s > 1 or per_nnz_img * int(rowptr[-1]) <= target:
            m_s = L.M
        else:
            frac = target / (per_nnz_img * int(rowptr[-1]))
            m_s = max(1, min(L.M, int(L.M * frac)))
    nnz_s = int(rowptr[m_s])
    xs = x[:n_s]
    args = (rowptr[:m_s + 1], colidx[:nnz_s], value[:nnz_s], m_s, L.R, L.S, L.stride, L.pad)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.csr(xs, *args)
        times.append(time.perf_counter() - t0)
    t_step = statistics.mean(times)
    scale = (int(rowptr[-1]) * L.N) / max(nnz_s * n_s, 1)
    us_layer = t_step * scale * 1e6
    sample = (f"oracle_csr (fp64) on images [0,{n_s}) x output channels [0,{m_s}) of "
              f"{L.name} ({nnz_s * n_s} of {int(rowptr[-1]) * L.N} nonzero-image pairs), "
              f"scaled to one layer; {steps} timed repeat(s)")
    return us_layer, threads, sample, times


def run_reference(args, L):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    rowptr, colidx, value = workloads.make_weights(L)
    x = workloads.make_input(L)
    budget = min(120.0, max(5.0, 0.02 * (args.steps + args.warmup)))
    # warm-up repeats are untimed
    if args.warmup:
        time_oracle(L, rowptr, colidx, value, x, budget * args.warmup /
                    max(args.steps + args.warmup, 1), steps=1)
    us, threads, sample, times = time_oracle(L, rowptr, colidx, value, x, budget,
                                             steps=args.steps)
    nnz = int(rowptr[-1])
    num = layer_numbers(L, nnz)
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(L, args.fmt, args.timing),
        "dense_equiv_tflops": num["dense_flop"] / (us * 1e-6) / 1e12,
        "useful_gflops": num["useful_flop"] / (us * 1e-6) / 1e9,
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# The CUDA path
# --------------------------------------------------------------------------

def graph_time(swd, torch, L, w, x, y, rowptr, colidx, value, fmt, steps, stream, dev,
               sample_clocks=False, local=0):
    """K forwards back to back, replayed from CUDA graphs, each on its own copy
    of input, weights and output; the copies together exceed twice the L2, so
    no launch finds its data in L2.  CUDA events on the launching stream
    around the whole region.  Returns (total ms, copies, bytes per copy, wall
    seconds, clock record or None)."""
    info = w.info()
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (126 << 20))
    per_copy = (x.numel() + y.numel()) * 4 + int(info["device_bytes"])
    n_copies = int(max(2, min(512, math.ceil(2 * l2 / per_copy))))
    xs, ys, hs = [x], [y], [w]
    for _ in range(n_copies - 1):
        xs.append(x.clone())
        ys.append(torch.empty_like(y))
        hs.append(swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R,
                           S=L.S, stride=L.stride, pad=L.pad, stream=stream,
                           fmt=fmt, batch_hint=L.N))
    for i in range(n_copies):
        swd.forward(xs[i], hs[i], out=ys[i], stream=stream)
    torch.cuda.synchronize(dev)
    group = min(n_copies, steps)
    full, rem = divmod(steps, group)

    def capture(count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(count):
                swd.forward(xs[i], hs[i], out=ys[i], stream=stream)
        return g

    g_full = capture(group)
    g_rem = capture(rem) if rem else None
    g_full.replay()
    if g_rem is not None:
        g_rem.replay()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = None
    if sample_clocks:
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.25)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    t_start.record(stream)
    for _ in range(full):
        g_full.replay()
    if g_rem is not None:
        g_rem.replay()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    clk = clocks.stop() if clocks is not None else None
    total_ms = t_start.elapsed_time(t_end)
    del g_full, g_rem
    torch.cuda.synchronize(dev)
    for h in hs[1:]:
        h.close()
    return total_ms, n_copies, per_copy, wall, clk


def roofline_of(L, nnz, fmt, us_kernel, sm_count):
    """The roofline and in-core records of one launch of `us_kernel` µs."""
    num = layer_numbers(L, nnz, 4 if fmt == "packed32" else roofline.ENTRY_BYTES)
    peaks, peak_kind = measured_peaks()
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    p_fp32 = fp32_peak_flops(sm_count, mhz)
    bw = float(peaks["hbm_gbs"]) * 1e9
    t_comp = num["useful_flop"] / p_fp32
    t_comm = num["alg_bytes"] / bw
    if t_comp >= t_comm:
        achieved = num["useful_flop"] / (us_kernel * 1e-6) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": p_fp32 / 1e12, "unit": "TFLOP/s",
                "frac": achieved / (p_fp32 / 1e12),
                "peak_source": f"{sm_count} SMs x 128 fp32 lanes x 2 x "
                               f"{mhz:.0f} MHz ({peak_kind} clock)"}
    else:
        achieved = num["alg_bytes"] / (us_kernel * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": bw / 1e9, "unit": "GB/s",
                "frac": achieved / (bw / 1e9), "peak_source": f"hbm_gbs ({peak_kind})"}
    kname = "spconv_ws_kernel" if fmt == "ws" else "spconv_fwd_kernel"
    roof["traffic"] = recorded_traffic(L.name if fmt == "f32" else f"{L.name}:{fmt}", kname)
    roof["algorithmic"] = num["alg_bytes"]
    roof["kernel"] = kname
    roof["roofline_us"] = max(t_comp, t_comm) * 1e6
    # Reported, not graded: the sparse path's in-core ceiling.  Every FMA of a
    # nonzero reads one 4-byte word of the staged input from shared memory,
    # which delivers 128 bytes per clock per SM: 32 FMAs per clock per SM, a
    # quarter of the fp32 rate.  (The dense-tap path reuses a register window
    # and is not bound by it; layers with many dense rows can exceed it.)
    p_smem = sm_count * 32 * 2 * mhz * 1e6
    in_core = {"ceiling": "shared memory, one 4-byte load per FMA of a nonzero",
               "achieved": num["useful_flop"] / (us_kernel * 1e-6) / 1e12,
               "peak": p_smem / 1e12, "unit": "TFLOP/s",
               "frac": num["useful_flop"] / (us_kernel * 1e-6) / p_smem,
               "peak_source": f"{sm_count} SMs x 128 B/clk / 4 B x 2 FLOP x {mhz:.0f} MHz"}
    return num, roof, in_core


# The other seeded layers the `layers` record times beside the headline one.
LAYER_SET = ("resnet3x3", "vgg3x3", "sweep50", "sweep80", "sweep90", "sweep95", "sweep99",
             "alex11x11", "conv5x5")


def time_layers(swd, torch, args, names, stream, dev, local, sm_count):
    """Each layer timed like the headline (graph replay over copies larger than
    L2, args.layer_steps steps), one entry per layer with its µs/layer,
    throughputs, roofline and in-core fractions and recorded DRAM traffic."""
    out = {}
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    for name in names:
        L = workloads.ALL_LAYERS[name]
        rowptr, colidx, value = workloads.make_weights(L)
        nnz = int(rowptr[-1])
        w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                     stride=L.stride, pad=L.pad, stream=stream, fmt=args.fmt, batch_hint=L.N)
        x = torch.from_numpy(workloads.make_input(L)).to(dev)
        y = torch.empty((L.N, L.M, L.E, L.F), device=dev, dtype=torch.float32)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                swd.forward(x, w, out=y, stream=stream)
            total_ms, n_copies, per_copy, _, _ = graph_time(
                swd, torch, L, w, x, y, rowptr, colidx, value, args.fmt, args.layer_steps,
                stream, dev)
        us = total_ms * 1e3 / args.layer_steps
        num, roof, in_core = roofline_of(L, nnz, args.fmt, us, sm_count)
        out[name] = {
            "value": us, "unit": UNIT, "steps": args.layer_steps,
            "config": describe(L, args.fmt, "graph"),
            "dense_equiv_tflops": num["dense_flop"] / (us * 1e-6) / 1e12,
            "useful_gflops": num["useful_flop"] / (us * 1e-6) / 1e9,
            "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                              "traffic", "algorithmic", "roofline_us")},
            "in_core": {"frac": in_core["frac"], "achieved": in_core["achieved"]},
            "nnz": nnz, "copies": n_copies,
            "launch": w.launch_info(L.N),
        }
        w.close()
        del x, y
        torch.cuda.synchronize(dev)
    clk = clocks.stop()
    return out, clk


def run_ours(args, L):
    import torch
    import torch.distributed as dist
    import sparse_weight_direct_gb300 as swd

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count

    rowptr, colidx, value = workloads.make_weights(L)
    x_host = workloads.make_input(L)
    nnz = int(rowptr[-1])
    stream = torch.cuda.Stream(device=dev)

    t0 = time.perf_counter()
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad, stream=stream, fmt=args.fmt, batch_hint=L.N)
    pack_ms = (time.perf_counter() - t0) * 1e3
    info = w.info()
    launch = w.launch_info(L.N)  # grid, cluster, reduction, shared memory of one launch

    x = torch.from_numpy(x_host).to(dev)
    y = torch.empty((L.N, L.M, L.E, L.F), device=dev, dtype=torch.float32)
    flush = torch.empty(FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
    x_pin = torch.from_numpy(x_host).pin_memory()
    y_pin = torch.empty(tuple(y.shape), dtype=torch.float32).pin_memory()
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            swd.forward(x, w, out=y, stream=stream)
        torch.cuda.synchronize(dev)

        # ---- latency of one launch after an L2 flush (events around each launch) ----
        lat_steps = args.steps if args.timing == "flush" else min(args.steps, 300)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(lat_steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(lat_steps)]
        if args.timing == "flush":
            clocks = ClockSampler(local)
            clocks.start()
            time.sleep(0.25)
        barrier()
        torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        for i in range(lat_steps):
            flush.zero_()
            starts[i].record(stream)
            swd.forward(x, w, out=y, stream=stream)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        per = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms
        if args.timing == "flush":
            wall = time.perf_counter() - wall0
            clk = clocks.stop()
            total_ms = sum(per)
            l2_detail = f"{lat_steps} launches, each after a 256 MiB write"
        else:
            # ---- throughput: the K steps back to back from CUDA graphs over
            # copies of the data larger than L2 ----
            barrier()
            total_ms, n_copies, per_copy, wall, clk = graph_time(
                swd, torch, L, w, x, y, rowptr, colidx, value, args.fmt, args.steps, stream,
                dev, sample_clocks=True, local=local)
            barrier()
            l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)
                     or (126 << 20))
            l2_detail = (f"{n_copies} copies of input, weights and output "
                         f"({n_copies * per_copy / 2**20:.0f} MiB; L2 {l2 / 2**20:.0f} MiB), "
                         f"the {args.steps} steps replayed back to back from CUDA graphs")

        # ---- end to end through the public API with host buffers ----
        e2e_steps = max(3, min(args.steps, 200))
        es = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
        for i in range(e2e_steps + 2):
            flush.zero_()
            if i >= 2:
                es[i - 2].record(stream)
            swd.forward_host(x_pin, w, y_pin, x, y, stream=stream)  # copy in, forward, copy out
            if i >= 2:
                ee[i - 2].record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = sum(s.elapsed_time(e) for s, e in zip(es, ee)) / e2e_steps

    # max over ranks
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], world, dev)

    ms_step = total_ms / args.steps
    us_layer = whole_job_us_per_layer(total_ms, args.steps, world)
    us_kernel = ms_step * 1e3                                 # one launch on one GPU
    num, roof, in_core = roofline_of(L, nnz, args.fmt, us_kernel, sm_count)

    line = {
        "metric": METRIC, "value": us_layer, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (fp16 weights)" if args.fmt == "packed32" else "f32", "data": "synthetic",
        "config": describe(L, args.fmt, args.timing),
        "timing": args.timing, "l2_detail": l2_detail,
        "dense_equiv_tflops": num["dense_flop"] / (us_kernel * 1e-6) / 1e12,
        "useful_gflops": num["useful_flop"] / (us_kernel * 1e-6) / 1e9,
        "alg_gbs": num["alg_bytes"] / (us_kernel * 1e-6) / 1e9,
        "us_per_launch": ms_step * 1e3,
        # one launch alone after an L2 flush, events around it (launch latency included)
        "latency_flushed_us": {"median": statistics.median(per) * 1e3,
                               "mean": statistics.fmean(per) * 1e3,
                               "sem": (statistics.stdev(per) / len(per) ** 0.5 * 1e3)
                               if len(per) > 1 else 0.0,
                               "steps": len(per)},
        "nnz": nnz, "pack_ms": pack_ms,
        "tiling": {**{k: info[k] for k in ("tile_rows", "lane_rows", "tiles_y", "tiles_x",
                                            "chunk", "num_chunks", "slots_per_warp", "groups",
                                            "blob_stride")},
                   "launch": launch},
        "roofline": roof,
        "in_core": in_core,
        "e2e": {"value": whole_job_us_per_layer(e2e_ms * e2e_steps, e2e_steps, world),
                "unit": UNIT,
                "h2d_bytes_per_step": int(x_host.nbytes),
                "d2h_bytes_per_step": int(y.numel() * 4)},
        "gpu_launches": args.steps,
        "clocks": clk,
        "wall_s": wall,
    }
    if args.compare_dense:
        # the dense library timed both ways, like the sparse kernel; the speedups
        # compare like with like (back to back: value; one launch alone: latency)
        dc = time_dense_conv(L, rowptr, colidx, value, x, y, flush, stream,
                             max(3, min(args.steps, 50)), args.timing == "graph")
        lat_us = statistics.fmean(per) * 1e3
        for key in ("fp32", "tf32"):
            if args.timing == "graph":
                dc[f"speedup_{key}"] = dc[f"{key}_graph_us"] / us_kernel
                dc[f"speedup_{key}_flushed"] = dc[f"{key}_us"] / lat_us
            else:
                dc[f"speedup_{key}"] = dc[f"{key}_us"] / us_kernel
        line["dense_conv"] = dc
    w.close()
    del x, y, flush
    torch.cuda.synchronize(dev)
    if rank == 0 and args.layers:
        # every other seeded layer, timed the same back-to-back way (outside the
        # headline's timed region)
        names = [n for n in LAYER_SET if n != L.name]
        layers, layer_clk = time_layers(swd, torch, args, names, stream, dev, local, sm_count)
        line["layers"] = layers
        line["layers_clocks"] = layer_clk
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        us_cpu, threads, sample, _ = time_oracle(L, rowptr, colidx, value, x_host,
                                                 budget_s=args.cpu_budget, steps=3)
        line["cpu_baseline"] = {"value": us_cpu, "unit": UNIT, "cores": threads,
                                "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def time_dense_conv(L, rowptr, colidx, value, x, y, flush, stream, steps, graph):
    """PyTorch's dense conv2d (cuDNN) on the same layer, the pages' baseline:
    fp32 with TF32 disabled, and PyTorch's default (TF32 allowed), each timed
    like the sparse kernel: one launch alone after an L2 flush (<key>_us) and,
    with graph, back to back from a CUDA graph over copies of its input and
    weights larger than L2 (<key>_graph_us).  Library run only."""
    import torch
    import torch.nn.functional as Fn
    w = np.zeros((L.M, L.CRS), dtype=np.float32)
    for m in range(L.M):
        w[m, colidx[rowptr[m]:rowptr[m + 1]]] = value[rowptr[m]:rowptr[m + 1]]
    wd = torch.from_numpy(w.reshape(L.M, L.C, L.R, L.S)).to(x.device)
    out = {}
    prev = torch.backends.cudnn.allow_tf32
    try:
        for key, tf32 in (("fp32", False), ("tf32", True)):
            torch.backends.cudnn.allow_tf32 = tf32
            with torch.cuda.stream(stream):
                for _ in range(3):
                    Fn.conv2d(x, wd, stride=L.stride, padding=L.pad)
                ts = []
                for _ in range(steps):
                    flush.zero_()
                    s0 = torch.cuda.Event(enable_timing=True)
                    s1 = torch.cuda.Event(enable_timing=True)
                    s0.record(stream)
                    Fn.conv2d(x, wd, stride=L.stride, padding=L.pad)
                    s1.record(stream)
                    ts.append((s0, s1))
                torch.cuda.synchronize()
                out[f"{key}_us"] = statistics.mean(a.elapsed_time(b) for a, b in ts) * 1e3
                if graph:
                    l2 = int(getattr(torch.cuda.get_device_properties(x.device), "L2_cache_size",
                                     0) or (126 << 20))
                    per_copy = (x.numel() + y.numel() + wd.numel()) * 4
                    n = int(max(2, min(512, math.ceil(2 * l2 / per_copy))))
                    xs = [x] + [x.clone() for _ in range(n - 1)]
                    ws = [wd] + [wd.clone() for _ in range(n - 1)]
                    for i in range(n):
                        Fn.conv2d(xs[i], ws[i], stride=L.stride, padding=L.pad)
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                        for i in range(n):
                            Fn.conv2d(xs[i], ws[i], stride=L.stride, padding=L.pad)
                    g.replay()
                    torch.cuda.synchronize()
                    reps = max(1, -(-steps // n))
                    s0 = torch.cuda.Event(enable_timing=True)
                    s1 = torch.cuda.Event(enable_timing=True)
                    s0.record(stream)
                    for _ in range(reps):
                        g.replay()
                    s1.record(stream)
                    torch.cuda.synchronize()
                    out[f"{key}_graph_us"] = s0.elapsed_time(s1) * 1e3 / (reps * n)
                    del g, xs, ws
                    torch.cuda.synchronize()
    finally:
        torch.backends.cudnn.allow_tf32 = prev
    out["library"] = f"torch {torch.__version__} cudnn {torch.backends.cudnn.version()}"
    return out


def run_timeline(args, L):
    """Per-block timeline of the forward kernel: needs the trace build
    (python sparse_weight_direct_gb300/build.py --trace, then
    SPCONV_LIBRARY=sparse_weight_direct_gb300/libspconv_trace.so).  Warm-up
    launches, then `steps` launches (at most 20), each after a 256 MiB L2 flush
    and timed alone; prints one JSON line summarising the launch with the
    median span: block durations by group kind, when each block's first stage
    was ready, how many blocks ran at once over time, and the blocks per SM.
    Not a benchmark line (the records cost a few stores per block)."""
    import numpy as np
    import torch
    import sparse_weight_direct_gb300 as swd
    from sparse_weight_direct_gb300 import _lib

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    rowptr, colidx, value = workloads.make_weights(L)
    stream = torch.cuda.Stream(device=dev)
    w = swd.pack(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                 stride=L.stride, pad=L.pad, stream=stream, fmt=args.fmt, batch_hint=L.N)
    launch = w.launch_info(L.N)
    nb = launch["grid_x"] * launch["grid_y"]
    x = torch.from_numpy(workloads.make_input(L)).to(dev)
    y = torch.empty((L.N, L.M, L.E, L.F), device=dev, dtype=torch.float32)
    flush = torch.empty(64 << 20, device=dev, dtype=torch.float32)
    buf = np.zeros(min(nb, 65536) * 4, dtype=np.uint64)
    lib = _lib.lib()
    runs = []
    for i in range(args.warmup + min(args.steps, 20)):
        flush.zero_()
        torch.cuda.synchronize()
        swd.forward(x, w, out=y, stream=stream)
        torch.cuda.synchronize()
        rc = lib.spconv_trace_read(buf.ctypes.data, buf.nbytes)
        if rc == _lib.SPCONV_ERR_UNSUPPORTED:
            print(json.dumps({"timeline": L.name, "error": "not the trace build: run "
                              "`python sparse_weight_direct_gb300/build.py --trace` and set "
                              "SPCONV_LIBRARY=sparse_weight_direct_gb300/libspconv_trace.so"}))
            return 1
        _lib.check(rc, "spconv_trace_read")
        if i >= args.warmup:
            runs.append(buf.reshape(-1, 4).astype(np.int64).copy())
    assert w.device_status(stream) == 0
    w.close()
    spans = [(r[:, 2].max() - r[:, 0].min()) / 1e3 for r in runs]
    rec = runs[int(np.argsort(spans)[len(spans) // 2])]
    if args.timeline_out:  # the raw records of that launch (uint64, blocks x 4)
        np.save(args.timeline_out, rec.astype(np.uint64))
    t0 = rec[:, 0].min()
    start, end = (rec[:, 0] - t0) / 1e3, (rec[:, 2] - t0) / 1e3
    ready = (rec[:, 1] - rec[:, 0]) / 1e3
    dur = end - start
    sm = rec[:, 3] & 0xFFFF
    flags = (rec[:, 3] >> 32) & 0xFF
    span = float(end.max())
    step = max(span / 20.0, 1e-3)
    ticks = np.arange(0.0, span, step)
    running = [int(((start <= t) & (end > t)).sum()) for t in ticks]
    peak = max(running) if running else 0
    half = next((float(t) for t, n in zip(ticks[1:], running[1:]) if n < peak / 2), span)

    def stats(a):
        return [round(float(a.min()), 2), round(float(np.median(a)), 2), round(float(a.max()), 2)]

    kinds = {}
    for name, m in (("dense", (flags & 1) != 0), ("split", (flags & 3) == 2),
                    ("sparse", (flags & 3) == 0)):
        if m.any():
            kinds[name] = {"blocks": int(m.sum()), "us_min_med_max": stats(dur[m]),
                           "end_max_us": round(float(end[m].max()), 2)}
    per_sm = np.bincount(sm, minlength=int(sm.max()) + 1)
    per_sm = per_sm[per_sm > 0]
    print(json.dumps({
        "timeline": L.name, "launches": len(runs), "blocks": int(nb),
        "grid": [launch["grid_x"], launch["grid_y"]], "cluster": launch["cluster"],
        "span_us": round(span, 2), "span_us_all_launches": [round(float(v), 2) for v in spans],
        "block_us_min_med_max": stats(dur), "by_kind": kinds,
        "first_stage_ready_us_med_max": [round(float(np.median(ready)), 2),
                                         round(float(ready.max()), 2)],
        "peak_running_blocks": peak,
        "ideal_span_us": round(float(dur.sum()) / max(peak, 1), 2),
        "below_half_peak_from_us": round(half, 2),
        "running_blocks_every_us": round(step, 2), "running_blocks": running,
        "blocks_per_sm_min_max": [int(per_sm.min()), int(per_sm.max())],
        "sms_used": int(per_sm.size)}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default=workloads.BENCH_DEFAULT,
                    choices=sorted(workloads.ALL_LAYERS))
    ap.add_argument("--timing", default="graph", choices=["graph", "flush"],
                    help="graph: the K steps back to back from CUDA graphs over copies of the "
                         "data larger than L2 (throughput); flush: each step timed alone "
                         "after an L2 flush (latency, launch overhead included)")
    ap.add_argument("--fmt", default="f32", choices=["f32", "packed32", "ws"],
                    help="packed weight format (packed32: the first page's 32-bit words, "
                         "FP16; ws: the weight-stationary mapping, one output channel per "
                         "block)")
    ap.add_argument("--compare-dense", action="store_true",
                    help="also time PyTorch's dense conv2d (cuDNN) on the same layer")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-layers", dest="layers", action="store_false",
                    help="skip the `layers` record (every other seeded layer timed the same "
                         "back-to-back way after the headline)")
    ap.add_argument("--layer-steps", type=int, default=0,
                    help="steps per layer of the `layers` record (default: max(steps, 20))")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline leg")
    ap.add_argument("--timeline", action="store_true",
                    help="per-block timeline of the forward kernel (trace build only; "
                         "see run_timeline)")
    ap.add_argument("--timeline-out", default="",
                    help="with --timeline: also save the median launch's raw records "
                         "(.npy, blocks x 4 uint64)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.layer_steps <= 0:
        args.layer_steps = max(args.steps, 20)
    L = workloads.ALL_LAYERS[args.config]
    if args.impl == "reference":
        return run_reference(args, L)
    if args.timeline:
        return run_timeline(args, L)
    return run_ours(args, L)


if __name__ == "__main__":
    sys.exit(main())
