#!/usr/bin/env python3
"""MXFP8 quantize benchmark: prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload fc1_8192x28672|act_4096x4096|grad_16384x8192|moe_64x65536x7168]

A step is one bidirectional (rowwise + colwise) quantize of the whole
workload, inputs already resident in device memory.  The metric is effective
bandwidth: (2 + 1 + 1 + 1/16) * M * N bytes per step (read BF16, write two FP8
planes and two E8M0 scale planes; + 4N for dbias) over the device-timed step.

Under torchrun (N > 1) every rank quantizes its own copy of the workload
(weak scaling, no collective on the data path); the timed region is
bracketed by barriers and the max over ranks is reported.

--impl reference times the CPU oracle (the only other implementation there
is) on a bounded sample of the same workload per step (32 rows per host core,
one thread per 32-row slice), on rank 0.  `cpu_baseline` times it the same way
on every host core, and single-threaded.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MXFP8 quantize effective GB/s and % of GB300 HBM peak (rowwise+colwise)"
BYTES_PER_ELEM = 2 + 1 + 1 + 1 / 16
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
# Every source the kernels are built from: a committed ncu traffic figure is only reported
# while these are unchanged since it was taken.
KERNEL_SOURCES = [f"mxfp8_block_scaled_04_gb300/csrc/{f}"
                  for f in ("api.cu", "dact.cuh", "dbias_reduce.cuh", "dgated.cuh", "ptx.cuh", "quantize.cuh")]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="fc1_8192x28672")
    ap.add_argument("--shape", default=None, help="MxN: the workload's value recipe at another shape")
    ap.add_argument("--swizzled", action="store_true", help="write GEMM-ready (swizzled) scale planes")
    ap.add_argument("--amax", action="store_true", help="also write the per-tensor amax")
    ap.add_argument("--dbias", action="store_true", help="fused dbias (per expert for the grouped workload)")
    ap.add_argument("--act", default="none", help="activation before the cast: relu, srelu, gelu, silu, qgelu")
    ap.add_argument("--dact", default="none",
                    help="backward fusion: quantize dY * act'(X), dY = the workload, X = N(0,1) of the same shape")
    ap.add_argument("--glu", default="none",
                    help="gated activation act(a) * b before the cast: x = [a | b] with a = the workload and "
                         "b = N(0,1) of the same shape (relu, srelu, gelu, silu = SwiGLU, qgelu)")
    ap.add_argument("--dglu", default="none",
                    help="gated backward: quantize [g b act'(a) | g act(a)] with g = the workload and "
                         "x = [a | b] two N(0,1) matrices of its shape (relu, srelu, gelu, silu, qgelu)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    return ap.parse_args()


def parse_shape(s):
    if not s:
        return None
    m, n = s.lower().split("x")
    return int(m), int(n)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def all_ranks_max(value: float, dist=None, device="cpu") -> float:
    """Max of a per-rank scalar over all ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_step: float, steps: int, world: int, total_ms: float) -> float:
    """Whole-job effective GB/s: every rank moved bytes_per_step per step in total_ms (the slowest rank)."""
    return bytes_per_step * steps * world / (total_ms / 1e3) / 1e9


def kernel_source_sha():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_name(args, M, N, workload_dbias):
    """Name of the committed ncu summary (profiles/<name>.md) for this run's kernel, workload and options."""
    name = args.workload if not args.shape else f"{args.workload.split('_')[0]}_{M}x{N}"
    family = ("quantize_dact" if args.dact.lower() != "none" else
              "quantize_gated" if args.glu.lower() != "none" else
              "quantize_dgated" if args.dglu.lower() != "none" else "quantize")
    opts = [o for o, on in (("swizzled", args.swizzled), ("amax", args.amax),
                            ("dbias", args.dbias and not workload_dbias)) if on]
    opts += [a.lower() for a in (args.act, args.dact, args.glu, args.dglu) if a.lower() != "none"]
    return "_".join([family, name] + opts)


def profiled_traffic(name):
    """DRAM bytes per step from the committed ncu summary, if it matches the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_step:\s*([0-9]+)", text)
    if not (m_sha and m_b) or m_sha.group(1) != kernel_source_sha():
        return None
    return int(m_b.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms in a background process."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid=None):
        self.samples = []   # (host time, sm, max, power, reasons)
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if gpu_uuid:
            cmd += ["-i", gpu_uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm, mx, pw = float(parts[0]), float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = [n for n, v in zip(names, parts[3:7]) if v.lower().startswith("active")]
            self.samples.append((time.time(), sm, mx, pw, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1, load_t0=None):
        inside = [s for s in self.samples if t0 <= s[0] <= t1 + 0.05]
        window = "timed region"
        if len(inside) < 3 and load_t0 is not None:
            inside = [s for s in self.samples if load_t0 <= s[0] <= t1 + 0.05]
            window = ("continuous load: the second half of the warm-up and the timed region "
                      "(timed region shorter than 3 sampling periods)")
        if not inside:
            inside, window = self.samples, "whole run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({r for s in inside for r in s[4]})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max(s[3] for s in inside)}


BAD_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def host_cores():
    """Cores this process may run on (the container's share, not the machine's count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_on_cores(oracle, x, fmt, threads):
    """Run the oracle over x split into `threads` contiguous 32-row slices, one per thread (the C
    oracle runs outside the GIL); returns the wall time."""
    from concurrent.futures import ThreadPoolExecutor

    stripes = x.shape[0] // 32
    bounds = [32 * (stripes * k // threads) for k in range(threads + 1)]
    parts = [x[bounds[k]:bounds[k + 1]] for k in range(threads) if bounds[k + 1] > bounds[k]]
    with ThreadPoolExecutor(max_workers=len(parts)) as pool:
        t = time.perf_counter()
        list(pool.map(lambda part: oracle.quantize(part, fmt), parts))
        return time.perf_counter() - t


def cpu_baseline(wl_x, N, fmt, target_s):
    """Time the oracle on the first rows of the workload: single-threaded, then on every host core
    (row slices per thread); each leg sized for about target_s / 2 of wall time."""
    import numpy as np
    import oracle

    oracle.build()
    cores = host_cores()
    stripe = np.ascontiguousarray(wl_x[:32])
    t = time.perf_counter()
    oracle.quantize(stripe, fmt)
    per_stripe = max(time.perf_counter() - t, 1e-6)
    max_stripes = wl_x.shape[0] // 32
    s1 = int(max(1, min(max_stripes, 0.5 * target_s / per_stripe)))
    sample1 = np.ascontiguousarray(wl_x[: 32 * s1])
    t = time.perf_counter()
    oracle.quantize(sample1, fmt)
    dt1 = time.perf_counter() - t
    single = BYTES_PER_ELEM * sample1.size / dt1 / 1e9
    sp = int(max(cores, min(max_stripes, 0.5 * target_s / per_stripe * cores)))
    sample_p = np.ascontiguousarray(wl_x[: 32 * sp])
    dtp = oracle_on_cores(oracle, sample_p, fmt, cores)
    return {"value": BYTES_PER_ELEM * sample_p.size / dtp / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {32 * sp} rows x {N} columns ({sample_p.size} elements) of the workload, scalar C "
                      f"oracle on {cores} threads (contiguous 32-row slices), {dtp:.2f} s",
            "single_thread": {"value": single, "unit": "GB/s", "cores": 1,
                              "sample": f"first {32 * s1} rows ({sample1.size} elements), {dt1:.2f} s"}}


def run_reference(args):
    """--impl reference: the CPU oracle, rank 0 only, bounded sample per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from mxfp8_block_scaled_04_gb300 import workloads as wl

    oracle.build()
    spec = wl.WORKLOADS[args.workload]
    M, N, fmt = spec[0], spec[1], spec[2]
    # sample: rows 0..31 of a workload-shaped input, C columns (C adaptive: whole run within ~2 minutes)
    full = wl.make(args.workload) if M * N <= 300_000_000 else None
    if full is None:
        raise SystemExit("workload too large for the reference arm")
    x = full["x"]
    cores = host_cores()
    probe = np.ascontiguousarray(x[:32, : min(N, 1024)])
    t = time.perf_counter()
    oracle.quantize(probe, fmt)
    per_elem = (time.perf_counter() - t) / probe.size
    # each step: 32 rows per core x C columns, one 32-row slice per thread
    budget = 120.0 / max(1, args.steps + args.warmup)
    C = int(max(32, min(N, (budget / per_elem / 32) // 32 * 32)))
    rows = min(32 * cores, M // 32 * 32)
    sample = np.ascontiguousarray(x[:rows, :C])
    threads = rows // 32
    for _ in range(args.warmup):
        oracle_on_cores(oracle, sample, fmt, threads)
    dt = 0.0
    for _ in range(args.steps):
        dt += oracle_on_cores(oracle, sample, fmt, threads)
    value = BYTES_PER_ELEM * sample.size * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "fmt": "e4m3" if fmt == 0 else "e5m2",
                   "sample_per_step": f"rows 0..{rows - 1} x columns 0..{C - 1}"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} x {C} elements of the workload per step, scalar C oracle on "
                                   f"{threads} threads (one 32-row slice each)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def host_link_ceiling(h2d_bytes, d2h_bytes, reps=5):
    """Pinned host <-> device copy rates in this run: H2D alone, D2H alone, and both at once on
    two streams (bytes over the link / time), each the best of `reps` on buffers of the e2e step's
    sizes.  This is the ceiling the host-buffer path (e2e) runs against."""
    import torch

    hs = torch.empty(h2d_bytes, dtype=torch.uint8, pin_memory=True)
    hd = torch.empty(d2h_bytes, dtype=torch.uint8, pin_memory=True)
    ds = torch.empty(h2d_bytes, dtype=torch.uint8, device="cuda")
    dd = torch.empty(d2h_bytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def best(fn, nbytes):
        out = 0.0
        for _ in range(reps):
            torch.cuda.synchronize()
            t = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            out = max(out, nbytes / (time.perf_counter() - t) / 1e9)
        return out

    def both():
        with torch.cuda.stream(s1):
            ds.copy_(hs, non_blocking=True)
        with torch.cuda.stream(s2):
            hd.copy_(dd, non_blocking=True)

    r = {"h2d_gbs": best(lambda: ds.copy_(hs, non_blocking=True), h2d_bytes),
         "d2h_gbs": best(lambda: hd.copy_(dd, non_blocking=True), d2h_bytes),
         "both_gbs": best(both, h2d_bytes + d2h_bytes),
         "how": "pinned copies of the e2e step's sizes, best of %d, wall clock around synchronize" % reps}
    del hs, hd, ds, dd
    return r


def run_ours(args):
    import numpy as np
    import torch

    import mxfp8_block_scaled_04_gb300 as mx
    from mxfp8_block_scaled_04_gb300 import workloads as wl

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    w = wl.make(args.workload, shape=parse_shape(args.shape))
    x_bits, fmt, with_dbias, offsets = w["x"], w["fmt"], w["with_dbias"] or args.dbias, w["offsets"]
    M, N = x_bits.shape
    grouped = offsets is not None
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    dglu = mx.binding.ACTIVATIONS[args.dglu.lower()]
    W = 2 if dglu else 1    # the gated backward writes [da | db]: outputs of width 2N
    out_row = torch.empty((M, W * N), dtype=torch.uint8, device="cuda")
    layout = mx.SCALES_SWIZZLED if args.swizzled else mx.SCALES_PLAIN
    if grouped and args.swizzled:   # one GEMM-ready plane per group
        row_bytes = mx.mxfp8_grouped_swizzled_scale_bytes(offsets, N, False)
        col_bytes = mx.mxfp8_grouped_swizzled_scale_bytes(offsets, N, True)
    else:
        row_bytes = mx.mxfp8_scale_bytes(M, W * (N // 32), layout)
        col_bytes = mx.mxfp8_scale_bytes(W * N, M // 32, layout)
    scale_row = torch.empty((row_bytes,), dtype=torch.uint8, device="cuda")
    out_col = torch.empty((M, W * N), dtype=torch.uint8, device="cuda")
    scale_col = torch.empty((col_bytes,), dtype=torch.uint8, device="cuda")
    amax = torch.empty((1,), dtype=torch.float32, device="cuda") if args.amax else None
    act = mx.binding.ACTIVATIONS[args.act.lower()]
    dact = mx.binding.ACTIVATIONS[args.dact.lower()]
    if dact and (act or args.swizzled or args.amax or grouped):
        raise SystemExit("--dact takes a flat workload without --act / --swizzled / --amax")
    x_act = (torch.from_numpy(wl.normal_bf16(M, N, seed=1234).view(np.int16)).view(torch.bfloat16).cuda()
             if dact else None)
    glu = mx.binding.ACTIVATIONS[args.glu.lower()]
    x_in_bits = x_bits
    x_gate = None
    if dglu:
        if act or dact or glu or args.swizzled or args.amax or grouped or with_dbias:
            raise SystemExit("--dglu takes a flat workload without dbias or other options")
        xg_bits = np.ascontiguousarray(np.concatenate([wl.normal_bf16(M, N, seed=1234),
                                                       wl.normal_bf16(M, N, seed=4321)], axis=1))
        x_gate = torch.from_numpy(xg_bits.view(np.int16)).view(torch.bfloat16).cuda()
    if glu:
        if act or dact or args.swizzled or args.amax or with_dbias:
            raise SystemExit("--glu takes a workload without dbias or other options")
        x_in_bits = np.ascontiguousarray(np.concatenate([x_bits, wl.normal_bf16(M, N, seed=4321)], axis=1))
        x = torch.from_numpy(x_in_bits.view(np.int16)).view(torch.bfloat16).cuda()
    if args.amax and offsets is not None:
        raise SystemExit("--amax applies to the flat workloads")
    if args.swizzled and grouped and (glu or with_dbias):
        raise SystemExit("--swizzled on the grouped workload takes no --glu / --dbias")
    if act and with_dbias:
        raise SystemExit("--act does not combine with the dbias workload")
    G = offsets.size - 1 if grouped else 0
    dbias = (torch.empty((G, N) if grouped else (N,), dtype=torch.float32, device="cuda") if with_dbias else None)
    ws_bytes = (mx.mxfp8_quantize_grouped_dbias_workspace_bytes(M, N, G) if grouped
                else mx.mxfp8_quantize_workspace_bytes(M, N, True))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if with_dbias else None
    off_dev = torch.from_numpy(offsets).cuda() if grouped else None
    stream = torch.cuda.current_stream()

    def step(xin=x):
        if grouped and args.swizzled:
            st = mx.mxfp8_quantize_grouped_swizzled(xin, M, N, G, off_dev, fmt, act, out_row, scale_row, out_col,
                                                    scale_col, None, None, stream)
        elif grouped and glu:
            st = mx.mxfp8_quantize_gated_grouped(xin, M, N, G, off_dev, fmt, glu, out_row, scale_row, out_col,
                                                 scale_col, None, None, stream)
        elif grouped and act:
            st = mx.mxfp8_quantize_grouped_activated(xin, M, N, G, off_dev, fmt, act, out_row, scale_row, out_col,
                                                     scale_col, None, None, stream)
        elif grouped and with_dbias:
            st = mx.mxfp8_quantize_grouped_dbias(xin, M, N, G, off_dev, fmt, out_row, scale_row, out_col,
                                                 scale_col, dbias, ws, None, None, stream)
        elif grouped:
            st = mx.mxfp8_quantize_grouped(xin, M, N, G, off_dev, fmt, out_row, scale_row,
                                           out_col, scale_col, None, None, None, stream)
        elif dact:
            st = mx.mxfp8_quantize_dact(xin, x_act, M, N, fmt, dact, out_row, scale_row, out_col, scale_col,
                                        dbias, ws, None, stream)
        elif glu:
            st = mx.mxfp8_quantize_gated(xin, M, N, fmt, glu, out_row, scale_row, out_col, scale_col, None, stream)
        elif dglu:
            st = mx.mxfp8_quantize_dgated(xin, x_gate, M, N, fmt, dglu, out_row, scale_row, out_col, scale_col,
                                          None, stream)
        elif args.swizzled or args.amax or act:
            cfg = mx.make_config(xin, M, N, fmt, out_row, scale_row, out_col, scale_col, dbias, ws, None,
                                 layout, amax, act)
            st = mx.mxfp8_quantize_ex(cfg, stream)
        else:
            st = mx.mxfp8_quantize(xin, M, N, fmt, out_row, scale_row, out_col, scale_col, dbias, ws, None,
                                   stream)
        if st != 0:
            raise mx.MXFP8Error(st, "bench step")

    algo_bytes = ((BYTES_PER_ELEM + (2 if dact or glu else 0)) * M * N if not dglu else
                  (3 * 2 + 2 * (1 + 1 + 1 / 16)) * M * N) + (4 * N * max(G, 1) if with_dbias else 0)
    prof = profile_name(args, M, N, w["with_dbias"])
    kernels = (["amax_init_kernel"] if args.amax else []) + ["quantize_dact_kernel" if dact or glu else "quantize_dgated_kernel" if dglu else "quantize_kernel"]
    if with_dbias:
        kernels.append("dbias_reduce_grouped_kernel" if grouped else "dbias_reduce_kernel")
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None

    # Clock sampling runs from the start of the warm-up.  Warm-up: at least W steps,
    # continued until 300 ms have passed so that the clocks have left their idle
    # state (measured: the first ~50 calls after idle run a few percent slow); the
    # timed region follows it at once, with no idle gap.
    sampler = ClockSampler(uuid)
    warm_t0 = time.perf_counter()
    warm_wall0 = time.time()
    warmup_run = 0
    while warmup_run < max(3, args.warmup) or time.perf_counter() - warm_t0 < 0.3:
        step()
        warmup_run += 1
        if warmup_run % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()

    # Inputs that fit in L2 would be re-read from L2 on the next step:
    # flush L2 (write a 256 MiB buffer) before every timed step and time only the steps.
    flush = M * N * 2 <= L2_BYTES
    flush_buf = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device="cuda") if flush else None

    def timed():
        # Per-step events only when L2 is flushed between steps (the flush must stay outside
        # the timed intervals); otherwise two events bracket the K back-to-back steps, and a
        # step's average duration is total / K (gaps between launches included).
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] if flush else None
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] if flush else None
        t_begin = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        launches0 = mx.mxfp8_kernel_launch_count()
        barrier()
        torch.cuda.synchronize()
        h0 = time.time()
        t_begin.record(stream)
        for i in range(args.steps):
            if flush:
                flush_buf.zero_()
                starts[i].record(stream)
            step()
            if flush:
                ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        h1 = time.time()
        barrier()
        launches = mx.mxfp8_kernel_launch_count() - launches0
        if flush:
            per_launch = [s.elapsed_time(e) for s, e in zip(starts, ends)]
            total_ms = sum(per_launch)
        else:
            total_ms = t_begin.elapsed_time(t_end)
            per_launch = [total_ms / args.steps]
        return total_ms, per_launch, launches, h0, h1

    total_ms, per_launch, launches, h0, h1 = timed()
    # a timed region shorter than the sampling period is judged with the samples of the
    # continuous load around it: the second half of the warm-up and the timed region
    clocks = sampler.summary(h0, h1, warm_wall0 + 0.15)
    if BAD_REASONS & set(clocks.get("reasons", [])):
        for _ in range(16):
            step()
        torch.cuda.synchronize()
        total_ms, per_launch, launches, h0, h1 = timed()     # re-measure once
        clocks = sampler.summary(h0, h1, h0 - 0.05)
        clocks["remeasured"] = True
    sampler.stop()

    # Host cost of one call: wall time of enqueueing back-to-back calls with no
    # synchronisation in between (the GPU runs behind; 64 calls stay far below
    # the launch queue's depth).
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(64):
        step()
    host_us = (time.perf_counter() - t0) / 64 * 1e6
    torch.cuda.synchronize()

    total_ms = all_ranks_max(total_ms, dist, "cuda")
    ms_per_step = total_ms / args.steps
    value = aggregate_gbs(algo_bytes, args.steps, world, total_ms)
    kernel_ms = statistics.mean(per_launch)
    peak, peak_src = measured_peak()
    achieved = algo_bytes / (kernel_ms / 1e3) / 1e9

    # ---- end to end through the public API: pinned host in, pinned host out ----
    e2e = None
    if not args.no_e2e:
        x_host = torch.from_numpy(x_in_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        outs_dev = [out_row, scale_row, out_col, scale_col] + ([dbias] if with_dbias else []) + \
            ([amax] if amax is not None else [])
        outs_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs_dev]
        h2d = x_host.numel() * 2
        d2h = sum(t.numel() * t.element_size() for t in outs_host)
        second = x_act if dact else x_gate if dglu else None   # the two-input calls' other input
        second_host = second.cpu().pin_memory() if second is not None else None
        if second_host is not None:
            h2d += second_host.numel() * 2
        if grouped and not (with_dbias or args.swizzled or glu):
            staging = torch.empty(mx.mxfp8_quantize_grouped_host_staging_bytes(M, N, G), dtype=torch.uint8,
                                  device="cuda")
            off_host = torch.from_numpy(offsets.astype(np.int64))
            path = ("mxfp8_quantize_grouped_host: pinned host buffers in and out, host offsets, H2D / kernel / "
                    "D2H pipelined over row chunks inside the library")

            def e2e_step():
                st = mx.mxfp8_quantize_grouped_host(x_host, M, N, G, off_host, fmt, act, *outs_host[:4], staging,
                                                    staging.numel(), stream)
                if st != 0:
                    raise mx.MXFP8Error(st, "bench e2e step")
        elif (dact or glu or dglu) and not grouped:
            if dact:
                nbytes = mx.mxfp8_quantize_dact_host_staging_bytes(M, N, with_dbias)
                name = "mxfp8_quantize_dact_host"
            elif glu:
                nbytes = mx.mxfp8_quantize_gated_host_staging_bytes(M, N)
                name = "mxfp8_quantize_gated_host"
            else:
                nbytes = mx.mxfp8_quantize_dgated_host_staging_bytes(M, N)
                name = "mxfp8_quantize_dgated_host"
            staging = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
            path = (f"{name}: pinned host buffers in and out (every input), H2D / kernel / D2H pipelined over "
                    "row chunks inside the library")

            def e2e_step():
                if dact:
                    st = mx.mxfp8_quantize_dact_host(x_host, second_host, M, N, fmt, dact, *outs_host[:4],
                                                     outs_host[4] if with_dbias else None, staging, staging.numel(),
                                                     stream)
                elif glu:
                    st = mx.mxfp8_quantize_gated_host(x_host, M, N, fmt, glu, *outs_host[:4], staging,
                                                      staging.numel(), stream)
                else:
                    st = mx.mxfp8_quantize_dgated_host(x_host, second_host, M, N, fmt, dglu, *outs_host[:4], staging,
                                                       staging.numel(), stream)
                if st != 0:
                    raise mx.MXFP8Error(st, "bench e2e step")
        elif (args.swizzled or args.amax or act) and not (grouped or dact or glu or dglu):
            amax_host = outs_host[-1] if amax is not None else None
            cfg_host = mx.make_config(x_host, M, N, fmt, *outs_host[:4], outs_host[4] if with_dbias else None, None,
                                      None, layout, amax_host, act)
            staging = torch.empty(mx.mxfp8_quantize_ex_host_staging_bytes(cfg_host), dtype=torch.uint8,
                                  device="cuda")
            path = ("mxfp8_quantize_ex_host: pinned host buffers in and out, H2D / kernel / D2H pipelined over "
                    "row chunks inside the library")

            def e2e_step():
                st = mx.mxfp8_quantize_ex_host(cfg_host, staging, staging.numel(), stream)
                if st != 0:
                    raise mx.MXFP8Error(st, "bench e2e step")
        elif grouped or args.swizzled or args.amax or act or dact or glu or dglu:
            # no host-buffer call for these options: copy in, device call, copy every output out
            x_stage = torch.empty_like(x)
            path = "pinned host -> device copy, C-ABI call, device -> pinned host copies (one stream)"

            def e2e_step():
                x_stage.copy_(x_host, non_blocking=True)
                step(x_stage)
                for hd, dd in zip(outs_host, outs_dev):
                    hd.copy_(dd, non_blocking=True)
        else:
            staging = torch.empty(mx.mxfp8_quantize_host_staging_bytes(M, N, with_dbias), dtype=torch.uint8,
                                  device="cuda")
            path = ("mxfp8_quantize_host: pinned host buffers in and out, H2D / kernel / D2H pipelined over "
                    "row chunks inside the library")

            def e2e_step():
                st = mx.mxfp8_quantize_host(x_host, M, N, fmt, *outs_host[:4],
                                            outs_host[4] if with_dbias else None, staging, staging.numel(),
                                            stream)
                if st != 0:
                    raise mx.MXFP8Error(st, "bench e2e step")

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(3, args.e2e_steps)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = all_ranks_max(a.elapsed_time(b) / n_e2e, dist, "cuda")
        link = host_link_ceiling(h2d, d2h)
        link_gbs = (h2d + d2h) / (e2e_ms / 1e3) / 1e9
        e2e = {"value": aggregate_gbs(algo_bytes, 1, world, e2e_ms), "unit": "GB/s", "ms_per_step": e2e_ms,
               "steps": n_e2e, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "path": path,
               "host_link_gbs": link_gbs, "host_link_ceiling": link,
               "frac_of_link_ceiling": link_gbs / link["both_gbs"]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x_bits, N, fmt, args.cpu_seconds)

    fault = mx.mxfp8_device_fault_word()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "warmup_steps_run": warmup_run, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload + (f"@{M}x{N}" if args.shape else ""), "M": M, "N": N, "fmt": "e4m3" if fmt == 0 else "e5m2",
                       "directions": "rowwise+colwise", "dbias": with_dbias, "grouped": grouped,
                       "scales": "swizzled" if args.swizzled else "plain", "amax": bool(args.amax),
                       "activation": args.act.lower(), "dact": args.dact.lower(), "glu": args.glu.lower(), "dglu": args.dglu.lower(),
                       "bytes_per_step": algo_bytes,
                       "l2": (f"L2 flushed (256 MiB written) before each timed step; {M * N * 2 / 1e6:.0f} MB "
                              f"bf16 input; time = sum of the per-step event intervals" if flush else
                              f"inputs larger than L2: {M * N * 2 / 1e6:.0f} MB bf16 read per step vs "
                              f"{L2_BYTES / 2 ** 20:.0f} MiB L2, no flush"),
                       "parallelism": f"{world} independent replica(s)" if world > 1 else "single GPU"},
            "pct_of_8tbs": 100 * value / world / 8000.0,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": f"{peak_src} hbm_gbs",
                         "traffic": profiled_traffic(prof),
                         "traffic_source": f"profiles/{prof}.md",
                         "kernel": " + ".join(kernels),
                         "kernel_ms": kernel_ms, "algorithmic_bytes_per_launch": algo_bytes},
            "clocks": clocks,
            "host_us_per_call": host_us,
            "gpu_launches": launches,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "device_fault_word": fault,
            "kernel_source_sha": kernel_source_sha(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        from mxfp8_block_scaled_04_gb300 import build

        if build.needs_build():
            build.build()
        run_ours(args)


if __name__ == "__main__":
    main()
