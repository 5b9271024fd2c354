"""Benchmark: NVFP4 row-scaled quantize-transpose of linear-layer operands.

One step = the whole hot path over one batch: for the activation X (16384 x 8192
BF16) and the gradient dY (16384 x 28672 BF16), the fused exact row+column amax
pass followed by the encode pass that writes rowwise and columnwise E2M1 codes
and E4M3 scales (row-scaled: rows use the row amax, columns the column amax).

The step is issued as nvfp4_amax + nvfp4_quantize_both(amax_in = that amax) per
operand -- the same kernels nvfp4_quantize_both launches on its own (prep, amax,
encode; with four-over-six one encode pass per direction) -- so that CUDA events
on the launching stream can time the encode pass alone for the roofline figure.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("NVFP4 quantize-transpose GB/s (BF16 in + codes/scales out) and % of GB300 HBM peak")
ROWS, K_X, K_DY = 16384, 8192, 28672
WORKLOAD = ("linear-layer operands: X 16384x8192 and dY 16384x28672 BF16, N(0,0.02) x per-row "
            "LogNormal(0,1); row-scaled NVFP4 quantize, fused row+col amax, rowwise+columnwise "
            "1x16 E2M1/E4M3 outputs, bound 448")


def bytes_io(rows, cols):
    """BF16 in once + codes + scales (both directions) + amax out."""
    codes = rows * ((cols + 1) // 2) + cols * ((rows + 1) // 2)
    scales = rows * ((cols + 15) // 16) + cols * ((rows + 15) // 16)
    return 2 * rows * cols + codes + scales + 4 * (rows + cols)


def quant_bytes(rows, cols, elem=2, row_scaled=True):
    """B_io of one two-direction quantize call: x (elem bytes per value) in once, codes
    and scales of both directions out, and the amax written (a float per line
    row-scaled, one per direction per-tensor)."""
    amax = 4 * (rows + cols) if row_scaled else 8
    return bytes_io(rows, cols) - 4 * (rows + cols) + amax + (elem - 2) * rows * cols


def bytes_min(rows, cols):
    """B_io plus the second read of x that a global amax forces (x exceeds on-chip storage)."""
    return bytes_io(rows, cols) + 2 * rows * cols


def encode_bytes(rows, cols):
    """Algorithmic bytes of one encode-kernel launch: x once, codes+scales out, amax in."""
    return bytes_io(rows, cols)


# DRAM bytes (read + write) per launch of the encode kernel on this workload, mean of
# the X and dY launches, from one ncu capture of a full step (dram__bytes_read.sum +
# dram__bytes_write.sum, L2 left as the step leaves it).  To be taken again whenever
# the encode kernel changes.
ENCODE_TRAFFIC_BYTES = (361.4e6 + 1383.6e6) / 2


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "of measured"
    return 6800.0, "of fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.first = threading.Event()
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        # nvidia-smi takes a moment to start: the timed region begins once it samples
        self.first.wait(timeout=10.0)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())
            self.first.set()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(t_local: float, world: int, units_per_rank_step: float, steps: int,
                   device=None):
    """(slowest rank's time, whole-job rate): every rank processes the same units per
    step (independent replicas), and the job is done when the slowest rank is."""
    t_max = max_over_ranks(t_local, world, device)
    return t_max, world * units_per_rank_step * steps / t_max


# ---------------------------------------------------------------- CPU oracle leg

def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def timed_strips(jobs, threads: int, min_seconds: float):
    """Run the callables in `jobs` (one per row strip) on `threads` host threads, all
    of them once per round, rounds repeated until at least min_seconds have passed.
    The oracle's C calls release the GIL, so the strips run on separate cores.
    Returns (seconds, rounds)."""
    import concurrent.futures as cf
    rounds, t0 = 0, time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while True:
            list(ex.map(lambda f: f(), jobs))
            rounds += 1
            dt = time.perf_counter() - t0
            if dt >= min_seconds:
                return dt, rounds


def prepare_oracle_sample(strip_rows: int, threads: int = 1, seed: int = 2):
    """`threads` strips of `strip_rows` rows of X and dY (drawn from the same
    distribution on the CPU) and one job per strip: the single-threaded oracle on that
    strip, both directions, row-scaled (each strip's column amax is over its own rows,
    as a data-parallel rank's would be).  Returns (jobs, B_io bytes per round, what)."""
    import numpy as np
    import torch

    import oracle
    import workloads
    g = workloads.generator(seed, "cpu")
    rows = strip_rows * threads
    xs = [workloads.row_lognormal(rows, k, g, "cpu") for k in (K_X, K_DY)]
    bits = [x.view(torch.int16).numpy().view(np.uint16) for x in xs]

    def job(i):
        parts = [b[i * strip_rows:(i + 1) * strip_rows] for b in bits]
        return lambda: [oracle.quantize(p, "bf16", mode=oracle.ROW_SCALED, bound=448.0)
                        for p in parts]

    nbytes = threads * sum(bytes_io(strip_rows, k) for k in (K_X, K_DY))
    what = (f"{threads} strip(s) of {strip_rows} rows of X and dY, both directions, one "
            f"thread per strip")
    return [job(i) for i in range(threads)], nbytes, what


def oracle_sample(strip_rows: int, threads: int = 1, min_seconds: float = 0.0, seed: int = 2):
    """The cpu_baseline object (GB/s of B_io over the rows processed) of the oracle on
    prepare_oracle_sample's strips, repeated until min_seconds have passed."""
    jobs, nbytes, what = prepare_oracle_sample(strip_rows, threads, seed)
    dt, rounds = timed_strips(jobs, threads, min_seconds)
    return {"value": rounds * nbytes / dt / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle", "sample": f"{what}, {rounds} round(s)", "seconds": dt}


def headline_cpu_baseline(args):
    """The oracle on all host cores (one row strip per core), and on one core."""
    cores = host_cores()
    allc = oracle_sample(args.oracle_rows or 256, threads=cores, min_seconds=10.0)
    allc["single_core"] = oracle_sample(args.oracle_rows or 256, threads=1, min_seconds=5.0)
    return allc


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cores = host_cores()
    # one step: every core quantizes its own strip of the workload's rows once
    jobs, nbytes, what = prepare_oracle_sample(args.oracle_rows or 64, threads=cores)
    for _ in range(args.warmup):
        timed_strips(jobs, cores, 0.0)
    vals, t_all = [], []
    for _ in range(args.steps):
        dt, _ = timed_strips(jobs, cores, 0.0)
        vals.append(nbytes / dt / 1e9)
        t_all.append(dt)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(t_all), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": what},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": what},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ---------------------------------------------------------------- GPU leg

def run_ours(args):
    import torch

    import nvfp4_precision_quantization_gb300 as nv
    import workloads

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    nv.load_library()

    x, dy = workloads.linear(dev, rows=args.rows)
    ops = [x, dy]
    fos = args.workload == "linear-fos"
    cfg = nv.Config(nv.NVFP4_ROW_SCALED, 448.0, int(fos), 0)
    outs = []
    for t in ops:
        r, c = t.shape
        row = nv.alloc_out(r, c, r, dev)
        col = nv.alloc_out(c, r, c, dev)
        row.amax_in, col.amax_in = row.amax, col.amax
        outs.append((row, col))
    flush = l2_flush_buffer(dev)

    def step(ev=None):
        for i, (t, (row, col)) in enumerate(zip(ops, outs)):
            nv.nvfp4_amax(t, row.amax, col.amax, None, stream=stream)
            if ev is not None:
                ev[2 * i].record(stream)
            nv.nvfp4_quantize_both(t, cfg, row, col, stream=stream)
            if ev is not None:
                ev[2 * i + 1].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    mid = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_region = time.perf_counter()
    for k in range(K):
        flush.zero_()
        starts[k].record(stream)
        step(mid[k])
        ends[k].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_region = time.perf_counter() - t_region
    clocks = sampler.stop()
    clocks["timed_region_s"] = t_region

    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    shapes = [t.shape for t in ops]
    bio = sum(bytes_io(r, c) for r, c in shapes)
    t_total, rate = job_throughput(sum(step_ms) / 1e3, world, bio, K, dev)
    ms_per_step = 1e3 * t_total / K
    # encode-kernel durations (between the event after amax and after quantize)
    enc_x = [mid[k][0].elapsed_time(mid[k][1]) for k in range(K)]
    enc_dy = [(mid[k][2].elapsed_time(mid[k][3])) for k in range(K)]
    amax_x = [starts[k].elapsed_time(mid[k][0]) for k in range(K)]
    amax_dy = [mid[k][1].elapsed_time(mid[k][2]) for k in range(K)]

    bmin = sum(bytes_min(r, c) for r, c in shapes)
    elems = sum(r * c for r, c in shapes)
    value = rate / 1e9
    peak, peak_src = measured_peaks()
    enc_bytes = sum(encode_bytes(r, c) for r, c in shapes) / 2  # per launch (mean of the two)
    enc_dur = (statistics.mean(enc_x) + statistics.mean(enc_dy)) / 2 / 1e3
    achieved = enc_bytes / enc_dur / 1e9

    e2e = None if args.no_e2e else measure_e2e(nv, ops, outs, cfg, stream, dev, max(2, min(K, 5)))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = headline_cpu_baseline(args)

    if rank == 0:
        line = {
            "metric": METRIC if not fos else METRIC + ", four-over-six",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "pct_of_hbm_peak": 100.0 * value / world / peak,
            "config": {
                "workload": WORKLOAD + (", four-over-six (T in {6, 4} by squared error)"
                                        if fos else ""),
                "l2": "inputs larger than L2 (268 MB, 940 MB) and " + flush_note(flush),
                "input_sha256_first_64MiB": input_digest(x, dy),
                "bytes_io_per_step": bio, "bytes_min_per_step": bmin,
                "elements_per_step": elems,
                "gbps_bytes_min": world * bmin * K / t_total / 1e9,
                "pct_of_hbm_peak_bytes_min": 100.0 * bmin * K / t_total / 1e9 / peak,
                "elements_per_s": world * elems * K / t_total,
                "peak_gbs": peak, "peak_source": peak_src,
                "ms_amax_x": statistics.mean(amax_x), "ms_encode_x": statistics.mean(enc_x),
                "ms_amax_dy": statistics.mean(amax_dy), "ms_encode_dy": statistics.mean(enc_dy),
            },
            "roofline": {"kernel": "k_encode (encode pass)", "bound": "hbm",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_src,
                         "traffic": (ENCODE_TRAFFIC_BYTES if args.rows == ROWS and not fos
                                     else None),
                         "algorithmic_bytes": enc_bytes},
            "cpu_baseline": cpu,
            "e2e": e2e,
            # prep + amax + encode per operand; four-over-six encodes each direction
            # in its own pass
            "gpu_launches": (8 if fos else 6) * K,
            "clocks": clocks,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------- other rows of the path

SUPPLEMENTARY = {
    "weights16x16": "weights 8192x8192 BF16 N(0,0.02), per-tensor amax, 16x16 block scales, "
                    "rowwise + columnwise (tensor amax pass, then the encode pass)",
    "moe": "MoE tokens: 32 groups, counts Multinomial(65536, uniform), each zero-padded to a "
           "multiple of 128 rows, K 7168, N(0,1) BF16; grouped amax -> per-row expansion -> "
           "rowwise quantize, four-over-six, bound 256",
    "dequant": "dequantize of a row-scaled 4096x4096 quantization (0.1 % outliers x50): "
               "rowwise codes -> BF16 and columnwise codes -> FP32",
    "moe-col": "MoE tokens as above (padded), grouped columnwise for the weight-gradient "
               "GEMMs: each group's column amax over its rows, row-scaled, bound 448",
    "moe-ragged": "MoE tokens as above, quantized straight from the unpadded tokens into the "
                  "padded layout (padding rows not read): per-group amax, four-over-six, "
                  "bound 256, rowwise",
    "moe-gemm": "grouped NVFP4 GEMMs of the MoE layout (32 groups of Multinomial(65536) "
                "tokens, each padded to a multiple of 256 rows): per-expert fprop (tokens x "
                "K 7168, row-scaled, times 32 expert weights of N 2048, one amax per expert) "
                "and per-expert wgrad (dY^T [2048 x tokens] times X^T [7168 x tokens], "
                "columnwise, per-group column amax, K = each group's tokens); BF16 out; "
                "FLOPs over the padded rows",
    "rht": "random Hadamard transform of the wgrad operand dY 16384x28672 BF16 (per column, "
           "16-row blocks, (1/4) H16 diag(s), sign mask 0x6D2B) fused into its row-scaled "
           "columnwise quantize (per-column amax of the transform, bound 448)",
    "rht-both": "dY 16384x28672 BF16, row-scaled, both directions in one encode pass: rowwise "
                "as it is, columnwise after the random Hadamard transform (sign mask 0x6D2B); "
                "row amax of dY, column amax of the transform, bound 448",
    "outliers": "X 4096x4096 BF16 N(0,1), 0.1 % of the entries x50: per-tensor then "
                "row-scaled NVFP4 quantize, both directions, 1x16, bound 448 (each call: "
                "prep, amax pass, encode; X fits in L2, so its second read comes from L2)",
    "edge": "non-aligned 4000x5000 N(0,1), in BF16 and in FP32: row-scaled NVFP4 quantize, "
            "both directions, 1x16, bound 448 (direct stores: the pitches allow no sector "
            "or TMA stores)",
    "tiny": "X 256x256 BF16, N(0,1) x per-row factor log-uniform in [1e-2, 1e2]: row-scaled "
            "NVFP4 quantize, both directions, bound 448 (latency-bound)",
    "gemm": "NVFP4 GEMM consumer of the linear layer: fprop Y[16384x28672] = X[16384x8192] "
            "W[28672x8192]^T (X row-scaled, W per-tensor) and wgrad dW[28672x8192] = "
            "dY^T[28672x16384] X (both row-scaled: bilateral post-scale); random NVFP4 operand "
            "bytes, BF16 output",
}


# the transform's sign mask in the rht workload (the method's random signs, fixed)
RHT_SIGN_MASK = 0x6D2B


def supplementary_oracle_sample(w: str, strip_rows: int, min_seconds: float = 10.0,
                                threads: int = 1):
    """The oracle on `threads` strips of `strip_rows` rows of the workload's input, one
    host thread per strip (each runs the single-threaded oracle on its own strip), in
    the workload's unit (algorithmic GB/s of the rows processed).  All strips once make
    a round; rounds repeat until at least min_seconds have been timed."""
    import numpy as np
    import torch

    import oracle
    import workloads

    def bits(t):
        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), "bf16"
        return t.numpy(), "fp32"

    n = strip_rows * threads
    jobs, nbytes = [], 0
    if w in ("moe", "moe-ragged", "moe-col"):
        xb, _ = bits(workloads.seeded_normal(n, 7168, seed=workloads.SEEDS["moe"] + 1000))
        ends = np.array([strip_rows], np.int64)
        cols = 7168
        for i in range(threads):
            part = xb[i * strip_rows:(i + 1) * strip_rows]
            if w == "moe-col":
                jobs.append(lambda p=part: oracle.quantize(p, "bf16", mode=oracle.ROW_SCALED,
                                                           bound=448.0, rowwise=False))
            else:
                jobs.append(lambda p=part: oracle.grouped_quantize_rowwise(
                    p, "bf16", ends, mode=oracle.PER_TENSOR, bound=256.0, four_over_six=True))
        per = 2 * strip_rows * cols + strip_rows * cols // 2 + strip_rows * cols // 16
        per += 4 * (cols if w == "moe-col" else strip_rows)
        nbytes = threads * per
        what = f"{threads} strip(s) of {strip_rows} tokens x 7168 (one group each)"
    elif w == "rht":
        g = workloads.generator(workloads.SEEDS["linear"], "cpu")
        xb, _ = bits(workloads.row_lognormal(n, 28672, g, "cpu"))
        cols = 28672
        for i in range(threads):
            part = xb[i * strip_rows:(i + 1) * strip_rows]
            jobs.append(lambda p=part: oracle.quantize_columnwise_rht(
                p, "bf16", RHT_SIGN_MASK, mode=oracle.ROW_SCALED, bound=448.0))
        nbytes = threads * (2 * strip_rows * cols + strip_rows * cols // 2
                            + strip_rows * cols // 16 + 4 * cols)
        what = f"{threads} strip(s) of {strip_rows} rows (tokens) of a 28672-column dY"
    elif w == "rht-both":
        g = workloads.generator(workloads.SEEDS["linear"], "cpu")
        xb, _ = bits(workloads.row_lognormal(n, 28672, g, "cpu"))
        cols = 28672
        for i in range(threads):
            part = xb[i * strip_rows:(i + 1) * strip_rows]
            jobs.append(lambda p=part: (
                oracle.quantize(p, "bf16", mode=oracle.ROW_SCALED, bound=448.0,
                                columnwise=False),
                oracle.quantize_columnwise_rht(p, "bf16", RHT_SIGN_MASK, mode=oracle.ROW_SCALED,
                                               bound=448.0)))
        nbytes = threads * (2 * strip_rows * cols + 2 * (strip_rows * cols // 2
                                                          + strip_rows * cols // 16)
                            + 4 * (cols + strip_rows))
        what = (f"{threads} strip(s) of {strip_rows} rows (tokens) of a 28672-column dY, "
                f"both directions")
    elif w == "weights16x16":
        xb, _ = bits(workloads.edge_normal(n, 8192, torch.bfloat16, "cpu", std=0.02))
        cols = 8192
        for i in range(threads):
            part = xb[i * strip_rows:(i + 1) * strip_rows]
            jobs.append(lambda p=part: oracle.quantize(p, "bf16", mode=oracle.PER_TENSOR,
                                                       bound=448.0, block_2d=True))
        nbytes = threads * (2 * strip_rows * cols
                            + 2 * (strip_rows * cols // 2 + strip_rows * cols // 16) + 8)
        what = f"{threads} strip(s) of {strip_rows} rows of the 8192x8192 weights, both directions"
    elif w in ("outliers", "edge", "tiny"):
        if w == "outliers":
            srcs = [bits(workloads.outliers("cpu")[:n])]
            modes = (oracle.PER_TENSOR, oracle.ROW_SCALED)
        elif w == "edge":
            srcs = [bits(workloads.edge_normal(n, 5000, dt, "cpu"))
                    for dt in (torch.bfloat16, torch.float32)]
            modes = (oracle.ROW_SCALED,)
        else:
            srcs = [bits(workloads.tiny("cpu")[:n])]
            modes = (oracle.ROW_SCALED,)
        for i in range(threads):
            parts = [(xb[i * strip_rows:(i + 1) * strip_rows], tag) for xb, tag in srcs]
            jobs.append(lambda ps=parts: [oracle.quantize(p, tag, mode=m, bound=448.0)
                                          for p, tag in ps for m in modes])
        for xb, tag in srcs:
            for m in modes:
                nbytes += threads * quant_bytes(strip_rows, xb.shape[1], 2 if tag == "bf16" else 4,
                                                m == oracle.ROW_SCALED)
        what = (f"{threads} strip(s) of {strip_rows} rows of the workload's input, "
                "both directions")
    else:  # dequant
        xb, _ = bits(workloads.outliers("cpu")[:n])
        cols = 4096
        for i in range(threads):
            part = xb[i * strip_rows:(i + 1) * strip_rows]
            o = oracle.quantize(part, "bf16", mode=oracle.ROW_SCALED, bound=448.0,
                                columnwise=False)["row"]
            jobs.append(lambda o=o: oracle.dequantize(o[0], o[1], o[2], row_scaled=True,
                                                      rows=strip_rows, cols=cols, bound=448.0,
                                                      out_dtype="fp32"))
        nbytes = threads * (strip_rows * cols // 2 + strip_rows * cols // 16 + 4 * strip_rows
                            + 4 * strip_rows * cols)
        what = (f"{threads} strip(s) of {strip_rows} rows of the 4096x4096 rowwise "
                "quantization, to FP32")
    dt, rounds = timed_strips(jobs, threads, min_seconds)
    return {"value": rounds * nbytes / dt / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle", "sample": f"{what}, {rounds} round(s)", "seconds": dt}


# rows per host thread in the oracle samples of the other rows of the path (the
# 4096-row inputs are cut into as many strips as there are cores)
SUPPLEMENTARY_STRIP_ROWS = {"tiny": 16, "outliers": 256, "dequant": 256, "edge": 128}


def supplementary_cpu_baseline(w: str, args):
    """All host cores (one strip each); on the small configs a single core as well."""
    cores = host_cores()
    rows = args.oracle_rows or SUPPLEMENTARY_STRIP_ROWS.get(w, 256)
    if w in ("outliers", "dequant", "tiny"):
        total = {"tiny": 256}.get(w, 4096)
        rows = max(1, min(rows, total // cores))
    r = supplementary_oracle_sample(w, rows, min_seconds=10.0, threads=cores)
    if w in ("tiny", "outliers", "edge"):
        r["single_core"] = supplementary_oracle_sample(w, rows, min_seconds=5.0, threads=1)
    return r


def run_supplementary(args):
    """One JSON line for a row of the path other than the headline workload: same
    timing rules (warm-up, an L2 flush of twice the L2 before each step, CUDA events on the
    launching stream, clocks sampled during the timed region)."""
    import torch

    import nvfp4_precision_quantization_gb300 as nv
    import workloads

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    nv.load_library()
    w = args.workload
    if w == "weights16x16":
        x = workloads.edge_normal(8192, 8192, torch.bfloat16, dev, std=0.02)
        M, K = x.shape
        cfg = nv.Config(nv.NVFP4_PER_TENSOR, 448.0, 0, 1)
        t = torch.empty(1, dtype=torch.float32, device=dev)
        row, col = nv.alloc_out(M, K, 1, dev), nv.alloc_out(K, M, 1, dev)
        row.amax, col.amax, row.amax_in, col.amax_in = t, t, t, t

        def step(ev):
            nv.nvfp4_amax(x, tensor_amax=t, stream=stream)
            ev[0].record(stream)
            nv.nvfp4_quantize_both(x, cfg, row, col, stream=stream)
        bio = 2 * M * K + 2 * (M * K // 2 + M * K // 16) + 8
        bmin = bio + 2 * M * K
        kern, kbytes, launches = "k_encode (16x16)", bio - 4, 3
        dtype, elems = "bf16", M * K
    elif w == "moe":
        x, ends, _, _ = workloads.moe(dev)
        M, K = x.shape
        G = ends.numel()
        cfg = nv.Config(nv.NVFP4_ROW_SCALED, 256.0, 1, 0)
        row = nv.alloc_out(M, K, M, dev)
        gam = torch.empty(G, dtype=torch.float32, device=dev)

        def step(ev):
            # the kernels nvfp4_grouped_quantize_rowwise (per-group amax) launches:
            # group check, the tiled row amax, each group's max written back to its
            # rows, then the rowwise encode
            nv.nvfp4_grouped_amax(x, ends, gam, row_amax_expanded=row.amax, stream=stream)
            ev[0].record(stream)
            row.amax_in = row.amax
            nv.nvfp4_quantize_rowwise(x, cfg, row, stream=stream)
        bio = 2 * M * K + M * K // 2 + M * K // 16 + 4 * M + 4 * G
        # a group (about 29 MB) fits in L2, so the floor reads x from HBM once; these
        # kernels read it twice (the amax pass, then the encode pass)
        bmin = bio
        kern, kbytes, launches = "k_encode (rowwise, four-over-six)", bio - 4 * G, 4
        dtype, elems = "bf16", M * K
    elif w == "moe-col":
        x, ends, _, _ = workloads.moe(dev)
        M, K = x.shape
        G = ends.numel()
        cfg = nv.Config(nv.NVFP4_ROW_SCALED, 448.0, 0, 0)
        col = nv.alloc_out(K, M, G * K, dev)

        def step(ev):
            # the same launches as nvfp4_grouped_quantize_columnwise: check, the amax
            # pass publishing per group, then the columnwise encode
            ev[0].record(stream)
            nv.nvfp4_grouped_quantize_columnwise(x, ends, cfg, col, stream=stream)
        bio = 2 * M * K + M * K // 2 + M * K // 16 + 4 * G * K
        bmin = bio + 2 * M * K
        kern, kbytes, launches = "whole step (check, grouped column amax, encode)", bio, 3
        dtype, elems = "bf16", M * K
    elif w == "moe-ragged":
        xp, pad_ends, counts, padded = workloads.moe(dev)
        x, rag_ends = workloads.moe_ragged(xp, counts, padded)
        x, rag_ends = x.contiguous(), rag_ends.to(dev)
        del xp
        T, K = x.shape
        M = int(padded.sum())
        G = len(counts)
        cfg = nv.Config(nv.NVFP4_PER_TENSOR, 256.0, 1, 0)
        row = nv.alloc_out(M, K, M, dev)
        gam = torch.empty(G, dtype=torch.float32, device=dev)

        def step(ev):
            ev[0].record(stream)
            nv.nvfp4_grouped_quantize_rowwise_padded(x, rag_ends, pad_ends, M, cfg, row, gam,
                                                     stream=stream)
        bio = 2 * T * K + M * K // 2 + M * K // 16 + 4 * M + 4 * G
        bmin = bio  # as for the padded tokens: each group fits in L2
        kern, kbytes, launches = ("whole step (check, row amax, group reduce, expand, rowwise "
                                   "encode)"), bio, 5
        dtype, elems = "bf16", M * K
    elif w == "rht":
        x = workloads.linear(dev, rows=args.rows)[1]
        M, K = x.shape
        cfg = nv.Config(nv.NVFP4_ROW_SCALED, 448.0, 0, 0)
        col = nv.alloc_out(K, M, K, dev)

        def step(ev):
            ev[0].record(stream)
            nv.nvfp4_quantize_columnwise_rht(x, RHT_SIGN_MASK, cfg, col, stream=stream)
        bio = 2 * M * K + M * K // 2 + M * K // 16 + 4 * K
        # fused: the amax pass and the encode pass each read x and transform it
        bmin = bio + 2 * M * K
        kern, kbytes, launches = "whole step (prep, transformed column amax, encode)", bmin, 3
        dtype, elems = "bf16", M * K
    elif w == "rht-both":
        x = workloads.linear(dev, rows=args.rows)[1]
        M, K = x.shape
        cfg = nv.Config(nv.NVFP4_ROW_SCALED, 448.0, 0, 0)
        row = nv.alloc_out(M, K, M, dev)
        col = nv.alloc_out(K, M, K, dev)

        def step(ev):
            ev[0].record(stream)
            nv.nvfp4_quantize_both_rht(x, RHT_SIGN_MASK, cfg, row, col, stream=stream)
        bio = 2 * M * K + 2 * (M * K // 2 + M * K // 16) + 4 * (M + K)
        # x is read twice: one pass for x's row maxima and the transform's column
        # maxima, then the encode
        bmin = bio + 2 * M * K
        kern, kbytes, launches = ("whole step (prep, row and transformed column amax, "
                                  "encode)"), bmin, 3
        dtype, elems = "bf16", M * K
    elif w in ("outliers", "edge", "tiny"):
        if w == "outliers":
            xs = [workloads.outliers(dev)]
            modes = [nv.NVFP4_PER_TENSOR, nv.NVFP4_ROW_SCALED]
        elif w == "edge":
            xs = [workloads.edge_normal(4000, 5000, dt_, dev)
                  for dt_ in (torch.bfloat16, torch.float32)]
            modes = [nv.NVFP4_ROW_SCALED]
        else:
            xs = [workloads.tiny(dev)]
            modes = [nv.NVFP4_ROW_SCALED]
        calls = []
        for xx in xs:
            M, K = xx.shape
            for md in modes:
                rs_ = md == nv.NVFP4_ROW_SCALED
                calls.append((xx, nv.Config(md, 448.0, 0, 0),
                              nv.alloc_out(M, K, M if rs_ else 1, dev),
                              nv.alloc_out(K, M, K if rs_ else 1, dev),
                              quant_bytes(M, K, xx.element_size(), rs_)))

        def step(ev):
            # whole calls (prep, amax pass, encode each); ev[0] precedes the last one
            for j, (xx, cc, row_, col_, _) in enumerate(calls):
                if j == len(calls) - 1:
                    ev[0].record(stream)
                nv.nvfp4_quantize_both(xx, cc, row_, col_, stream=stream)
        bio = sum(c_[4] for c_ in calls)
        # the second read of x (the encode pass after the amax pass) stays in L2 here
        bmin = bio
        last = "FP32 " if w == "edge" else "row-scaled " if w == "outliers" else ""
        kern = f"whole {last}quantize call (prep, amax, encode)"
        kbytes, launches = calls[-1][4], 3 * len(calls)
        dtype = "bf16" if w != "edge" else "bf16, f32"
        elems = sum(c_[0].numel() for c_ in calls)
    elif w == "dequant":
        x = workloads.outliers(dev)
        M, K = x.shape
        cfg = nv.Config(nv.NVFP4_ROW_SCALED, 448.0, 0, 0)
        row, col = nv.alloc_out(M, K, M, dev), nv.alloc_out(K, M, K, dev)
        nv.nvfp4_quantize_both(x, cfg, row, col, stream=stream)
        out_bf16 = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        out_f32 = torch.empty(K, M, dtype=torch.float32, device=dev)

        def step(ev):
            nv.nvfp4_dequantize(row.codes, row.scales, row.amax, nv.NVFP4_ROW_SCALED, M, K, 448.0,
                                out_bf16, stream=stream)
            ev[0].record(stream)
            nv.nvfp4_dequantize(col.codes, col.scales, col.amax, nv.NVFP4_ROW_SCALED, K, M, 448.0,
                                out_f32, stream=stream)
        codes_scales = M * K // 2 + M * K // 16
        bio = (codes_scales + 4 * M + 2 * M * K) + (codes_scales + 4 * K + 4 * M * K)
        bmin = bio
        kern, kbytes, launches = "k_dequantize (FP32 out)", codes_scales + 4 * K + 4 * M * K, 2
        dtype, elems = "f32", 2 * M * K
    else:
        raise SystemExit(f"unknown workload {w}")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = supplementary_cpu_baseline(w, args)

    flush = l2_flush_buffer(dev)
    for _ in range(args.warmup):
        flush.zero_()
        step([torch.cuda.Event(enable_timing=True)])
    torch.cuda.synchronize()
    K_ = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K_)]
    ends_ = [torch.cuda.Event(enable_timing=True) for _ in range(K_)]
    mids = [[torch.cuda.Event(enable_timing=True)] for _ in range(K_)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_region = time.perf_counter()
    for k in range(K_):
        flush.zero_()
        starts[k].record(stream)
        step(mids[k])
        ends_[k].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_region = time.perf_counter() - t_region
    clocks = sampler.stop()
    clocks["timed_region_s"] = t_region
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends_)]
    t_total, rate = job_throughput(sum(step_ms) / 1e3, world, bio, K_, dev)
    kern_ms = statistics.mean(m[0].elapsed_time(e) for m, e in zip(mids, ends_))
    peak, peak_src = measured_peaks()
    achieved = kbytes / (kern_ms / 1e3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": f"NVFP4 {w} GB/s (algorithmic bytes in + out) and % of GB300 HBM peak",
            "value": rate / 1e9, "unit": "GB/s", "n_gpus": world, "steps": K_,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_total / K_, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "pct_of_hbm_peak": 100.0 * rate / 1e9 / world / peak,
            "config": {"workload": SUPPLEMENTARY[w],
                       "l2": flush_note(flush),
                       "bytes_io_per_step": bio, "bytes_min_per_step": bmin,
                       "gbps_bytes_min": world * bmin * K_ / t_total / 1e9,
                       "pct_of_hbm_peak_bytes_min": 100.0 * bmin * K_ / t_total / 1e9 / peak,
                       "elements_per_s": world * elems * K_ / t_total,
                       "peak_gbs": peak, "peak_source": peak_src},
            "roofline": {"kernel": kern, "bound": "hbm", "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_src,
                         "traffic": None, "algorithmic_bytes": kbytes},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": launches * K_,
            "clocks": clocks}))
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_e2e(nv, ops, outs, cfg, stream, dev, steps):
    """Same metric through the C ABI with host buffers: pinned H2D of X and dY, the
    quantize, D2H of codes, scales and amax, all inside the timed region.  Copies run
    on their own streams so that the transfers of one operand overlap the other's
    quantize and each other (host to device and device to host at once), as a
    training step would issue them; every byte still crosses inside the region."""
    import torch
    host_in = [t.cpu().pin_memory() for t in ops]
    host_out = []
    for row, col in outs:
        host_out.append([torch.empty_like(a, device="cpu").pin_memory()
                         for a in (row.codes, row.scales, row.amax, col.codes, col.scales,
                                   col.amax)])
    dev_in = [torch.empty_like(t) for t in ops]
    e2e_outs = []
    for t in ops:
        r, c = t.shape
        e2e_outs.append((nv.alloc_out(r, c, r, dev), nv.alloc_out(c, r, c, dev)))
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(a.numel() * a.element_size() for lst in host_out for a in lst)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    times = []
    for _ in range(steps + 1):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        copied = []
        for hi, di in zip(host_in, dev_in):  # all inputs in, in order
            with torch.cuda.stream(s_in):
                di.copy_(hi, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
            copied.append(ev)
        for di, (row, col), ho, ev in zip(dev_in, e2e_outs, host_out, copied):
            stream.wait_event(ev)
            nv.nvfp4_quantize_both(di, cfg, row, col, stream=stream)
            done = torch.cuda.Event()
            done.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                for dst, src in zip(ho, (row.codes, row.scales, row.amax, col.codes, col.scales,
                                         col.amax)):
                    dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        times.append(time.perf_counter() - t0)
    t = statistics.median(times[1:])
    bio = sum(bytes_io(*t_.shape) for t_ in ops)
    return {"value": bio / t / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * t,
            "overlap": "H2D, quantize and D2H on separate streams"}


# DRAM bytes (read + write) of the k_gemm_nvf4 launch of the wgrad call, from one ncu
# capture of the full-size step; to be taken again whenever the GEMM kernel changes.
GEMM_TRAFFIC_BYTES = 1962.3e6 + 516.5e6


def l2_flush_buffer(dev):
    """A buffer twice the device's L2 (from its properties), written before each timed
    step so that no step starts with the previous one's data in L2."""
    import torch
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20))
    return torch.empty(2 * l2, dtype=torch.uint8, device=dev)


def flush_note(flush) -> str:
    return f"a {flush.numel() / 2**20:.0f} MiB L2 flush (2x the device's L2) before each step"


def input_digest(*tensors, limit: int = 64 << 20) -> str:
    """SHA-256 of the first `limit` bytes of each synthetic input, concatenated (a
    fingerprint that the inputs are the seeded ones)."""
    import hashlib

    import torch
    h = hashlib.sha256()
    for t in tensors:
        b = t.reshape(-1).view(torch.uint8)[:limit]
        h.update(b.cpu().numpy().tobytes())
    return h.hexdigest()


def tensor_peak():
    """FP4 dense tensor peak: the measured BF16 burst GEMM rate times the nominal
    FP4 / BF16 ratio (13.5 / 2.25 = 6)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return 6.0 * float(json.load(open(p))["bf16_tflops"]), "of measured bf16 burst x 6"
    return 6.0 * 1900.0, "of fallback bf16 x 6"


def gemm_oracle_sample(lines: int, k: int):
    """The oracle's FP64 GEMM (single thread) on lines x lines outputs of depth k, in
    TFLOP/s of the products it forms."""
    import numpy as np

    import oracle
    import workloads
    ops = []
    for seed, rs in ((21, True), (22, False)):
        c, sc, a = workloads.nvfp4_operand(lines, k, seed, row_scaled=rs)
        ops.append(dict(codes=c.numpy(), scales=sc.numpy(), amax=a.numpy(), row_scaled=rs,
                        bound=448.0))
    t0 = time.perf_counter()
    oracle.gemm(ops[0], ops[1])
    dt = time.perf_counter() - t0
    return {"value": 2.0 * lines * lines * k / dt / 1e12, "unit": "TFLOP/s", "cores": 1,
            "kind": "oracle", "seconds": dt,
            "sample": f"{lines} x {lines} outputs of depth k = {k}, FP64"}


def run_gemm(args):
    """The GEMM consumer of the linear layer's NVFP4 operands: fprop Y = X W^T
    (X row-scaled, W per-tensor) and wgrad dW = dY^T X (both row-scaled: the
    bilateral post-scale), BF16 output; one step = both GEMMs."""
    import torch

    import nvfp4_precision_quantization_gb300 as nv
    import workloads

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    nv.load_library()
    calls, flops = [], 0
    grouped = args.workload == "moe-gemm"
    jobs = [("fprop", False), ("wgrad", True)]
    if args.gemm_shape:  # one GEMM of the given shape, both operands row-scaled
        jobs = [(tuple(args.gemm_shape), True)]
    if grouped:  # the MoE tokens (padded to 256 per group) and 32 experts
        _, _, pad_ends = workloads.moe_layout(align=256)
        groups, m, n, k = len(pad_ends), int(pad_ends[-1]), 2048, 7168
        ends = pad_ends.to(dev)
        # fprop: tokens [m][k] row-scaled x expert weights [groups*n][k], one amax per expert
        ca, sa, aa = workloads.nvfp4_operand(m, k, 41, row_scaled=True, device=dev)
        cb, sb, ab = workloads.nvfp4_operand(groups * n, k, 42, row_scaled=True, device=dev)
        a = nv.Operand(ca, sa, aa, nv.NVFP4_ROW_SCALED, 448.0)
        b = nv.Operand(cb, sb, ab[:groups].contiguous(), nv.NVFP4_PER_TENSOR, 448.0)
        d = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(nv.nvfp4_grouped_gemm_workspace_size(m, n, k, groups), dtype=torch.uint8,
                         device=dev)
        calls.append((a, b, d, ws, 2.0 * m * n * k, ("fprop", ends)))
        # wgrad: dY^T [n][tokens] x X^T [k][tokens], both columnwise, per-group column amax
        cg, sg, ag = workloads.nvfp4_operand(n, m, 43, row_scaled=True, device=dev)
        cx, sx, ax = workloads.nvfp4_operand(k, m, 44, row_scaled=True, device=dev)
        rng = torch.Generator(device=dev)
        rng.manual_seed(45)
        a2 = nv.Operand(cg, sg, torch.rand(groups * n, generator=rng, device=dev) + 0.5,
                        nv.NVFP4_ROW_SCALED, 448.0)
        b2 = nv.Operand(cx, sx, torch.rand(groups * k, generator=rng, device=dev) + 0.5,
                        nv.NVFP4_ROW_SCALED, 448.0)
        d2 = torch.empty(groups, n, k, dtype=torch.bfloat16, device=dev)
        ws2 = torch.empty(nv.nvfp4_gemm_workspace_size(n, k, m), dtype=torch.uint8, device=dev)
        calls.append((a2, b2, d2, ws2, 2.0 * n * k * m, ("wgrad", ends)))
        flops += 2.0 * m * n * k * 2
        jobs = []
    for i, (name, b_rs) in enumerate(jobs):
        m, n, k = name if isinstance(name, tuple) else workloads.GEMM_SHAPES[name]
        ca, sa, aa = workloads.nvfp4_operand(m, k, 31 + 2 * i, row_scaled=True, device=dev)
        cb, sb, ab = workloads.nvfp4_operand(n, k, 32 + 2 * i, row_scaled=b_rs, device=dev)
        a = nv.Operand(ca, sa, aa, nv.NVFP4_ROW_SCALED, 448.0)
        b = nv.Operand(cb, sb, ab, nv.NVFP4_ROW_SCALED if b_rs else nv.NVFP4_PER_TENSOR, 448.0)
        d = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(nv.nvfp4_gemm_workspace_size(m, n, k), dtype=torch.uint8, device=dev)
        calls.append((a, b, d, ws, 2.0 * m * n * k, None))
        flops += 2.0 * m * n * k

    def step(ev):
        for j, (a, b, d, ws, _, grp) in enumerate(calls):
            if j == len(calls) - 1:
                ev[0].record(stream)
            if grp is None:
                nv.nvfp4_gemm(a, b, d, ws, stream=stream)
            elif grp[0] == "fprop":
                nv.nvfp4_grouped_gemm(a, b, grp[1], d, ws, stream=stream)
            else:
                nv.nvfp4_grouped_gemm_wgrad(a, b, grp[1], d, ws, stream=stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = gemm_oracle_sample(args.oracle_rows or 512, 7168 if grouped else
                                 workloads.GEMM_SHAPES["fprop"][2])
    flush = l2_flush_buffer(dev)
    for _ in range(args.warmup):
        flush.zero_()
        step([torch.cuda.Event(enable_timing=True)])
    torch.cuda.synchronize()
    K_ = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K_)]
    ends_ = [torch.cuda.Event(enable_timing=True) for _ in range(K_)]
    mids = [[torch.cuda.Event(enable_timing=True)] for _ in range(K_)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_region = time.perf_counter()
    for k_ in range(K_):
        flush.zero_()
        starts[k_].record(stream)
        step(mids[k_])
        ends_[k_].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_region = time.perf_counter() - t_region
    clocks = sampler.stop()
    clocks["timed_region_s"] = t_region
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends_)]
    t_total, rate = job_throughput(sum(step_ms) / 1e3, world, flops, K_, dev)
    kern_ms = statistics.mean(m[0].elapsed_time(e) for m, e in zip(mids, ends_))
    peak, peak_src = tensor_peak()
    achieved = calls[-1][4] / (kern_ms / 1e3) / 1e12
    if rank == 0:
        print(json.dumps({
            "metric": "NVFP4 GEMM consumer TFLOP/s" + (
                " (grouped MoE fprop + wgrad)" if grouped else
                "" if args.gemm_shape else " (fprop + wgrad of the linear layer)"),
            "value": rate / 1e12, "unit": "TFLOP/s", "n_gpus": world, "steps": K_,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_total / K_, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e2m1 x e2m1 -> f32 acc, bf16 out",
            "data": "synthetic",
            "config": {"workload": SUPPLEMENTARY[args.workload] if not args.gemm_shape else
                       "one NVFP4 GEMM %dx%dx%d, both operands row-scaled" % tuple(args.gemm_shape),
                       "l2": flush_note(flush),
                       "flops_per_step": flops, "peak_tflops": peak, "peak_source": peak_src,
                       "pct_of_tensor_peak": 100.0 * rate / 1e12 / world / peak},
            "roofline": {"kernel": "k_gemm_nvf4, last call of the step (its event time includes "
                                   "the call's scale pre-pass)",
                         "bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_src,
                         "traffic": None if (args.gemm_shape or grouped) else GEMM_TRAFFIC_BYTES,
                         "traffic_unit": "DRAM bytes per launch of k_gemm_nvf4",
                         "algorithmic_flops": calls[-1][4]},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": 3 * len(calls) * K_,
            "clocks": clocks}))
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--oracle-rows", type=int, default=None,
                    help="rows of X and dY in the oracle sample (default 2560 for the CPU "
                         "baseline, about 10 s of one Grace core; 128 per step for "
                         "--impl reference; GEMM workloads: lines of each operand, "
                         "default 512)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--rows", type=int, default=ROWS,
                    help="rows of X and dY (default 16384; smaller only for profiling captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gemm-shape", type=int, nargs=3, metavar=("M", "N", "K"), default=None,
                    help="--workload gemm: one GEMM of this shape per step instead of the "
                         "linear layer's two (smaller only for profiling captures)")
    ap.add_argument("--workload", default="linear",
                    choices=["linear", "linear-fos", *SUPPLEMENTARY],
                    help="linear (default): the headline workload; the others measure the "
                         "remaining rows of the path (four-over-six, 16x16 weights, grouped "
                         "MoE, dequantize), one JSON line each")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in ("gemm", "moe-gemm"):
        run_gemm(args)
    elif args.workload in SUPPLEMENTARY:
        run_supplementary(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
