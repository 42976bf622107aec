#!/usr/bin/env python
"""Benchmark of the MXFP8 linear layer (dynamic activation quantize + block-scaled GEMM).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one mxfp8_linear call (the library's public entry point, through
the Python binding) on the prefill MLP-up workload: x bf16 [4096, 4096]
quantised to MXFP8 inside the call, weights E4M3 [14336, 4096] with E8M0
block scales, bf16 out [4096, 14336].  The call runs the quantize kernel, then
the tcgen05 GEMM with its bias/bf16 epilogue.  Inputs are resident in HBM; the
L2 is flushed (a 256 MiB write, then a 256 MiB read so that no dirty lines are
left) between timed steps, outside the timed events.
Prints one JSON line (rank 0).  Secondary figures: each kernel timed alone
(separate runs), the decode sweep (M = 1, 4, 16, 64; N = K = 4096) as HBM
GB/s, the other workloads, and the two-layer chain.

With N > 1 (torchrun) every rank runs the same workload on its own GPU
(independent replicas: the layer has no exchange step); value is the work of
all ranks over the slowest rank's time.

--impl reference times the CPU oracle (the plain fp64 numpy implementation in
oracle/) on all host cores (one single-threaded process per core, each on its
own rows of the workload), on bounded samples of the same workload.
"""

from __future__ import annotations

import os

# The CPU oracle runs as one single-threaded process per host core; pin
# numpy's BLAS to one thread per process before it loads (the spawned workers
# inherit this).
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mxfp8_block_scaled_02_gb300 import synth  # noqa: E402

METRIC = "MXFP8 linear TFLOP/s (quant+GEMM) and % of GB300 FP8 peak; decode HBM GB/s"
WORKLOAD = "prefill MLP-up M4096 N14336 K4096, bf16 x quantised in the step, no bias"
FP8_PER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor rate (4.5 / 2.25 PFLOP/s)
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_pair_prefill_up.traffic.txt")
GEMM_SOURCE = os.path.join(ROOT, "mxfp8_block_scaled_02_gb300", "csrc", "gemm_pair.cu")


def _dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


class L2Flush:
    """Evict the L2 between timed steps: write a buffer larger than the L2, then
    read another one, so that the write's dirty lines are written back here and
    not inside the next timed step."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        self.r.sum()


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _traffic_for_current_gemm():
    """Per-launch DRAM bytes from the committed ncu summary, if it matches gemm_pair.cu."""
    try:
        kv = dict(line.split("=", 1) for line in open(TRAFFIC_FILE).read().split() if "=" in line)
        src_hash = hashlib.sha256(open(GEMM_SOURCE, "rb").read()).hexdigest()[:16]
        if kv.get("source_sha256_16") != src_hash:
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (the job's time is its slowest rank's)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step: float, steps: int, world: int, max_total_ms: float) -> float:
    """Whole-job throughput: the work of all ranks over the slowest rank's time.

    Every rank runs the same step on its own GPU (independent replicas: the
    layer has no exchange step), so the job does world * steps steps.
    """
    return flops_per_step * world * steps / (max_total_ms * 1e-3) / 1e12


def _dev_bf16(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def _oracle_worker_init(x_bits, w_bits):
    """Spawned worker: quantise its sample of the weights once (set-up, not timed)."""
    global _W
    import oracle
    wq, ws = oracle.quantize(synth.bf16_bits_to_f64(w_bits))
    _W = (synth.bf16_bits_to_f64(x_bits), wq, ws)


def _oracle_worker_run(job):
    """Spawned worker: `reps` oracle quant+GEMM calls on this worker's rows
    (or until `min_seconds` have passed); returns the calls made."""
    import oracle
    row0, rows, reps, min_seconds = job
    x, wq, ws = _W
    xs = x[row0:row0 + rows]
    n, t0 = 0, time.perf_counter()
    while n < reps or time.perf_counter() - t0 < min_seconds:
        oracle.linear_bf16(xs, wq, ws)
        n += 1
    return n


class OraclePool:
    """The CPU oracle on every host core: one spawned, single-threaded process
    per core, each on its own rows of the workload (the rows of a linear layer
    are independent), all against the same sample of weight rows."""

    def __init__(self, p: synth.LinearProblem, rows_per_worker: int, cols: int):
        import multiprocessing as mp
        self.cores = max(1, os.cpu_count() or 1)
        self.rows, self.cols, self.K = rows_per_worker, cols, p.K
        nrows = min(p.M, self.rows * self.cores)
        ctx = mp.get_context("spawn")
        self.pool = ctx.Pool(self.cores, initializer=_oracle_worker_init,
                             initargs=(np.ascontiguousarray(p.x[0, :nrows]),
                                       np.ascontiguousarray(p.w[0, :cols])))
        self.jobs = [((i * self.rows) % nrows, self.rows) for i in range(self.cores)]
        self.pool.map(_oracle_worker_run, [(r0, n, 1, 0.0) for r0, n in self.jobs])  # warm

    def flops_per_call(self) -> float:
        return 2.0 * self.rows * self.cols * self.K

    def run(self, reps: int, min_seconds: float = 0.0):
        """Every worker makes >= reps calls (and runs >= min_seconds); returns
        (total calls, wall seconds)."""
        t0 = time.perf_counter()
        calls = self.pool.map(_oracle_worker_run, [(r0, n, reps, min_seconds) for r0, n in self.jobs])
        return sum(calls), time.perf_counter() - t0

    def close(self):
        self.pool.terminate()
        self.pool.join()


def _cpu_oracle_rate(pool: OraclePool, min_seconds: float):
    """Oracle quant+GEMM over all host cores, >= min_seconds; TFLOP/s and details."""
    calls, el = pool.run(1, min_seconds)
    return pool.flops_per_call() * calls / el / 1e12, el, calls


def run_reference(args):
    """--impl reference: the CPU oracle on all host cores, bounded samples of
    the same workload (each step: one oracle call per core, on its own rows)."""
    rank, world, _ = _dist_env()
    if rank != 0:
        return
    p = synth.prefill_up()
    rows, cols = 4, 256
    pool = OraclePool(p, rows, cols)
    for _ in range(args.warmup):
        pool.run(1)
    calls, el = pool.run(args.steps)
    pool.close()
    value = pool.flops_per_call() * calls / el / 1e12
    sample = (f"{pool.cores} processes x {rows} rows x {cols} output columns x K={p.K} of the workload "
              f"per step ({calls} oracle calls in {el:.1f} s)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded SplitMix64 generator)",
        "config": {"workload": WORKLOAD, "M": p.M, "N": p.N, "K": p.K, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": pool.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _time_calls(fn, flush, stream, steps):
    """Per-call device time (ms) of `fn`, L2 flushed between calls outside the
    events; returns the list of times."""
    evs = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        flush.zero_()
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def run_ours(args):
    from mxfp8_block_scaled_02_gb300 import build, ops
    rank, world, local_rank = _dist_env()
    p = synth.prefill_up()
    # The oracle's worker processes start before any GPU work (spawned, so
    # they would be safe later too) and run after the GPU part is done.
    pool = OraclePool(p, rows_per_worker=16, cols=1024) if rank == 0 else None
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    build.build()
    ops.load()

    M, N, K = p.M, p.N, p.K
    flops = p.flops
    x = _dev_bf16(p.x[0], dev)
    w = _dev_bf16(p.w[0], dev)
    wq, ws = ops.quantize(w)                    # weights quantised once (E4M3 + E8M0)
    pw = ops.process_weights(wq, ws)
    del w, wq, ws
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    wsp = torch.empty(ops.workspace_size(1, M, N, K, False), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def step():                                 # one public mxfp8_linear call
        ops.linear(x, pw, out=out, workspace=wsp)

    for _ in range(args.warmup):
        step()
        flush.zero_()
    ops.check()

    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    cvd = [c for c in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if c]
    clocks = ClockSampler(cvd[local_rank] if local_rank < len(cvd) else str(local_rank))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_wall = time.perf_counter()
    for i in range(n):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
        flush.zero_()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    ops.check()
    step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]
    total_ms = max_over_ranks(sum(step_ms), dev)
    ms_per_step = total_ms / n
    value = job_tflops(flops, n, world, total_ms)

    # Each kernel of the call timed alone, in separate runs (same inputs, same
    # flush): the quantiser into the packed operand layout, then the GEMM on
    # the packed operands.
    k_steps = min(max(n, 20), 200)
    x_q = torch.empty((1, M, K), dtype=torch.uint8, device=dev)
    sfa = torch.empty(ops.packed_sizes(1, M, K)[1], dtype=torch.uint8, device=dev)
    pa = ops.quantize_packed(x, 1, x_q=x_q, sf_packed=sfa)
    out3 = out.view(1, M, N)
    quant_ms = statistics.mean(_time_calls(lambda: ops.quantize_packed(x, 1, x_q=x_q, sf_packed=sfa),
                                           flush, stream, k_steps))
    gemm_ms = statistics.mean(_time_calls(lambda: ops.gemm_packed(pa, pw, out=out3), flush, stream,
                                          k_steps))
    # the floor of this timing method: a kernel that zeroes 256 bytes, timed
    # the same way (one call between events, L2 flushed before it)
    tiny = torch.empty(256, dtype=torch.uint8, device=dev)
    floor_ms = statistics.median(_time_calls(lambda: tiny.zero_(), flush, stream, k_steps))
    ops.check()

    peaks, peak_src = _peaks()
    fp8_peak = peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]) * FP8_PER_BF16
    hbm_peak = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    traffic = _traffic_for_current_gemm()
    quant_bytes = M * K * 2 + M * K + M * K // 32

    # End to end through the public call with host buffers: every step copies
    # its x from pinned host memory, runs mxfp8_linear and copies its result
    # back to pinned host memory.  Consecutive steps are pipelined over three
    # streams (the upload of step i+1 and the download of step i-1 overlap the
    # compute of step i), with two device buffers each for x and out.
    x_host = torch.from_numpy(p.x[0].view(np.int16)).view(torch.bfloat16).pin_memory()
    out_host = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    o_dev = [out, torch.empty_like(out)]
    s_up, s_cmp, s_dn = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(steps):
        up, cmp_, dn = [], [], []
        for i in range(steps):
            k = i % 2
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(cmp_[i - 2])      # x_dev[k] is free once step i-2 has computed
                x_dev[k].copy_(x_host, non_blocking=True)
                up.append(torch.cuda.Event())
                up[-1].record(s_up)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(up[i])
                if i >= 2:
                    s_cmp.wait_event(dn[i - 2])       # o_dev[k] is free once step i-2 is downloaded
                ops.linear(x_dev[k], pw, out=o_dev[k], workspace=wsp)
                cmp_.append(torch.cuda.Event())
                cmp_[-1].record(s_cmp)
            with torch.cuda.stream(s_dn):
                s_dn.wait_event(cmp_[i])
                out_host[k].copy_(o_dev[k], non_blocking=True)
                dn.append(torch.cuda.Event())
                dn[-1].record(s_dn)

    e2e_steps = max(3, min(n, 50))
    e2e_run(3)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    e2e_run(e2e_steps)
    b.record(s_dn)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b) / e2e_steps
    ops.check()
    del x_dev, o_dev, x_q, sfa, pa

    decode = _decode_sweep(ops, dev, flush, stream, steps=min(max(n, 20), 500))
    # the same kernel on the MLP-up weights (N = 14336, K = 4096, no bias)
    decode["N14336_K4096"] = _decode_sweep(ops, dev, flush, stream, steps=min(max(n, 20), 200), ms=(1, 16),
                                           problem=synth.prefill_up())
    # x handed over already quantised (E4M3 codes + row-major scales)
    decode["prequantized_x"] = _decode_sweep(ops, dev, flush, stream, steps=min(max(n, 20), 200),
                                             ms=(1, 16, 64), prequantized=True)
    others = _other_workloads(ops, dev, flush, stream, steps=min(max(n, 10), 100))
    others["two_layer_mlp_M4096"] = _two_layer_chain(ops, dev, flush, stream, pw, x,
                                                     steps=min(max(n, 10), 100))
    others["mxfp6_e2m3_weights"] = _fp6_workloads(ops, dev, flush, stream, x, "e2m3",
                                                  steps=min(max(n, 10), 100))
    others["medium_m_N4096_K4096"] = _medium_m(ops, dev, flush, stream, steps=min(max(n, 10), 100))

    line = None
    if rank == 0:
        cpu_rate, cpu_s, cpu_calls = _cpu_oracle_rate(pool, min_seconds=10.0)
        pool.close()
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": n, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 x e4m3 -> fp32 accumulate (MXFP8, E8M0 block scales), bf16 out",
            "data": "synthetic (seeded SplitMix64 generator; random-init weights)",
            "config": {"workload": WORKLOAD, "B": 1, "M": M, "N": N, "K": K,
                       "x": "bf16 N(0,1), 0.1% entries x100, 1% of 32-blocks zero",
                       "step": "one mxfp8_linear call (quantize kernel + GEMM kernel)",
                       "l2": "flushed between timed steps (256 MiB write then 256 MiB read, "
                             "outside the events)",
                       "parallelism": f"replicas x{world}"},
            "fp8_peak_fraction": value / fp8_peak,
            "fp8_nominal_fraction": value / 4500.0,
            "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak,
                         "unit": "TFLOP/s", "frac": gemm_tflops / fp8_peak, "traffic": traffic,
                         "kernel": "gemm_mxf8_pair_kernel (tcgen05.mma.cta_group::2 kind::mxf8f6f4 block_scale)",
                         "peak_source": f"{peak_src} bf16 burst x {FP8_PER_BF16:g} (nominal FP8/BF16)",
                         "frac_of_nominal_4500": gemm_tflops / 4500.0},
            "kernels": {"timing": "each kernel alone, separate runs, L2 flushed between calls",
                        "quantize_us": quant_ms * 1e3,
                        "quantize_gbs": quant_bytes / (quant_ms * 1e-3) / 1e9,
                        "quantize_hbm_frac": quant_bytes / (quant_ms * 1e-3) / 1e9 / hbm_peak,
                        "event_floor_us": floor_ms * 1e3,
                        "event_floor": "a 256-byte zeroing kernel timed the same way: the fixed part of "
                                       "every per-call time in this block",
                        "gemm_us": gemm_ms * 1e3, "gemm_tflops": gemm_tflops},
            "decode_hbm": decode,
            "other_workloads": others,
            "cpu_baseline": {"value": cpu_rate, "unit": "TFLOP/s", "cores": pool.cores, "kind": "oracle",
                             "sample": f"{pool.cores} processes x 16 rows x 1024 output columns x K={K}, "
                                       f"{cpu_calls} oracle calls in {cpu_s:.1f} s (fp64 numpy, "
                                       f"one single-threaded process per core)"},
            "e2e": {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2,
                    "ms_per_step": e2e_ms,
                    "pipelining": "upload, compute and download on three streams, two buffers each"},
            "gpu_launches": 2 * n,
            "clocks": clk,
            "wall_s_timed_region": t_wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return line


def _decode_sweep(ops, dev, flush, stream, steps, fmt="e4m3", ms=(1, 4, 16, 64), problem=None,
                  prequantized=False):
    """Decode M in {1, 4, 16, 64}, N = K = 4096 with bias: HBM GB/s of the layer
    (weights in ``fmt``: E4M3, or packed MXFP6 with 3/4 of the weight bytes).

    Steady state of a decode loop: a CUDA graph of R back-to-back calls, each on
    its own copy of the weights (R copies together exceed twice the L2, so every
    call reads its weights from HBM), replayed `steps` times; per-call time =
    graph time / R.  Also reported: one call alone after an L2 flush ("cold"),
    which includes the launch and the SM reconfiguration after the flush.
    ``problem`` replaces the decode weights and x (e.g. the MLP-up weights,
    N = 14336, taking x from its first rows); its bias may be None.
    ``prequantized`` hands the layer x as E4M3 codes and row-major scales
    (quantised once, before the graph) instead of bf16.
    """
    p = problem if problem is not None else synth.decode(64)
    w = _dev_bf16(p.w[0], dev)
    wq, ws = ops.quantize_weights(w, fmt)
    base = ops.process_weights(wq, ws, fmt)
    bias = None if p.bias is None else _dev_bf16(p.bias, dev)
    del w, wq, ws
    per_copy = base.w_packed.numel() + base.sf_packed.numel()
    R = int(np.ceil(2 * 129e6 / per_copy)) + 1
    pws = [base] + [ops.PackedWeights(base.w_packed.clone(), base.sf_packed.clone(), base.B, base.N,
                                      base.K, base.batched, base.fmt) for _ in range(R - 1)]
    peaks, _ = _peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])
    res = {"weight_copies": R, "timing": "CUDA graph of back-to-back calls over rotating weight copies",
           "weights": fmt}
    reps = max(3, min(steps, 200))
    side = torch.cuda.Stream()
    for M in ms:
        x = _dev_bf16(p.x[0, :M], dev)
        xs = None
        if prequantized:
            x, xs = ops.quantize(x)
        out = torch.empty((M, p.N), dtype=torch.bfloat16, device=dev)
        wsb = torch.empty(max(ops.workspace_size(1, M, p.N, p.K, prequantized), 1), dtype=torch.uint8,
                          device=dev)
        for pw in pws:                                   # warm-up outside capture
            ops.linear(x, pw, bias, x_scale=xs, out=out, workspace=wsb)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for pw in pws:
                ops.linear(x, pw, bias, x_scale=xs, out=out, workspace=wsb)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (reps * R)
        cold = _time_steps(lambda: ops.linear(x, base, bias, x_scale=xs, out=out, workspace=wsb), flush,
                           stream, min(steps, 50))
        x_bytes = M * p.K + M * p.K // 32 if prequantized else 2 * M * p.K
        nbytes = (base.w_packed.numel() + p.N * p.K // 32 + x_bytes + 2 * M * p.N
                  + (0 if p.bias is None else 2 * p.N))
        res[f"M{M}"] = {"us": us, "gbs": nbytes / (us * 1e-6) / 1e9,
                        "hbm_frac": nbytes / (us * 1e-6) / 1e9 / hbm, "cold_us": cold,
                        "bytes_per_call": nbytes}
        del g
    ops.check()
    return res


def _time_steps(fn, flush, stream, steps):
    for _ in range(3):
        fn()
        flush.zero_()
    evs = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        flush.zero_()
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3


def _other_workloads(ops, dev, flush, stream, steps):
    """The pre-quantised prefill (MLP-down) and the batched workload, each
    through mxfp8_linear, against the roofline that binds it."""
    peaks, _ = _peaks()
    hbm = peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])
    fp8 = peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]) * FP8_PER_BF16
    res = {}
    # prefill MLP-down, x handed over pre-quantised (row-major scales)
    p = synth.prefill_down()
    x_q, x_s = ops.quantize(_dev_bf16(p.x[0], dev))
    p.x = None
    wq, ws = ops.quantize(_dev_bf16(p.w[0], dev))
    pw = ops.process_weights(wq, ws)
    del wq, ws
    out = torch.empty((p.M, p.N), dtype=torch.bfloat16, device=dev)
    wsb = torch.empty(ops.workspace_size(1, p.M, p.N, p.K, True), dtype=torch.uint8, device=dev)
    us = _time_steps(lambda: ops.linear(x_q, pw, x_scale=x_s, out=out, workspace=wsb), flush, stream, steps)
    tf = p.flops / (us * 1e-6) / 1e12
    res["prefill_down_prequantized_M8192_N4096_K14336"] = {
        "us": us, "tflops": tf, "fp8_peak_frac": tf / fp8, "bound": "tensor"}
    del x_q, x_s, pw, out, wsb
    # batched: 16 x (512 x 512 x 7168), bf16 x quantised in the call
    p = synth.bmm()
    x = _dev_bf16(p.x, dev)
    wq, ws = ops.quantize(_dev_bf16(p.w, dev))
    pw = ops.process_weights(wq, ws)
    out = torch.empty((p.B, p.M, p.N), dtype=torch.bfloat16, device=dev)
    wsb = torch.empty(ops.workspace_size(p.B, p.M, p.N, p.K, False), dtype=torch.uint8, device=dev)
    us = _time_steps(lambda: ops.linear(x, pw, out=out, workspace=wsb), flush, stream, steps)
    nbytes = p.B * (p.M * p.K * 2 + p.N * p.K + p.N * p.K // 32 + p.M * p.N * 2)
    res["bmm_B16_M512_N512_K7168"] = {
        "us": us, "tflops": p.flops / (us * 1e-6) / 1e12, "gbs": nbytes / (us * 1e-6) / 1e9,
        "hbm_frac": nbytes / (us * 1e-6) / 1e9 / hbm, "bound": "hbm (x bf16 read once)"}
    # the same layer on the GEMM that quantises x itself (path 5, not the default)
    us = _time_steps(lambda: ops.linear(x, pw, out=out, workspace=wsb, path=5), flush, stream, steps)
    res["bmm_B16_M512_N512_K7168_fused_quantize_path5"] = {
        "us": us, "gbs": nbytes / (us * 1e-6) / 1e9, "hbm_frac": nbytes / (us * 1e-6) / 1e9 / hbm}
    ops.check()
    return res


def _medium_m(ops, dev, flush, stream, steps):
    """Prefill chunks of 128 / 256 / 512 tokens at N = K = 4096 (bf16 x, one
    call after an L2 flush): the library's choice (path 0: the small-M kernel
    at 128 rows, split K over CTA pairs at 256), split-K CTA pairs (path 4)
    and unsplit CTA pairs (path 3)."""
    p = synth.decode(64)       # N = K = 4096 weights and bias of the decode workload
    wq, ws = ops.quantize(_dev_bf16(p.w[0], dev))
    pw = ops.process_weights(wq, ws)
    bias = _dev_bf16(p.bias, dev)
    res = {}
    for M in (128, 256, 512):
        x = _dev_bf16(synth.to_bf16_bits(synth.normal(77 + M, M * p.K)).reshape(M, p.K), dev)
        out = torch.empty((M, p.N), dtype=torch.bfloat16, device=dev)
        wsb = torch.empty(ops.workspace_size(1, M, p.N, p.K, False), dtype=torch.uint8, device=dev)
        flops = 2.0 * M * p.N * p.K
        r = {}
        for name, path in (("automatic", 0), ("split_k", 4), ("unsplit_pairs", 3)):
            us = _time_steps(lambda: ops.linear(x, pw, bias, out=out, workspace=wsb, path=path), flush, stream,
                             steps)
            r[name] = {"us": us, "tflops": flops / (us * 1e-6) / 1e12}
        res[f"M{M}"] = r
    ops.check()
    return res


def _fp6_workloads(ops, dev, flush, stream, x, fmt, steps):
    """MXFP6 weights (the mxfp6 page's E2M3 / E3M2, packed to 6 bits): the
    decode sweep (M = 1, 16) and the prefill MLP-up step with the same bf16 x,
    weights quantised by the library from the same bf16 draws."""
    res = {"decode": _decode_sweep(ops, dev, flush, stream, steps=max(steps, 20), fmt=fmt, ms=(1, 16))}
    p = synth.prefill_up()
    wq, ws = ops.quantize_weights(_dev_bf16(p.w[0], dev), fmt)
    pw = ops.process_weights(wq, ws, fmt)
    del wq, ws
    out = torch.empty((p.M, p.N), dtype=torch.bfloat16, device=dev)
    wsb = torch.empty(ops.workspace_size(1, p.M, p.N, p.K, False), dtype=torch.uint8, device=dev)
    us = _time_steps(lambda: ops.linear(x, pw, out=out, workspace=wsb), flush, stream, steps)
    res["prefill_up_M4096_N14336_K4096"] = {"us": us, "tflops": p.flops / (us * 1e-6) / 1e12}
    ops.check()
    return res


def _two_layer_chain(ops, dev, flush, stream, pw_up, x, steps):
    """A prefill MLP step of two layers, up (M4096 N14336 K4096) then down
    (M4096 N4096 K14336), with bf16 x: (a) the bf16 chain, where the down
    layer quantises the up layer's bf16 output with the standalone kernel;
    (b) the quantised hand-off, where the up layer's epilogue writes its output
    as MXFP8 codes + packed scales and the down layer reads them directly."""
    p = synth.prefill_down()
    p.x = None
    wq, ws = ops.quantize(_dev_bf16(p.w[0], dev))
    pw_down = ops.process_weights(wq, ws)
    del wq, ws
    M = x.shape[0]
    h = torch.empty((M, pw_up.N), dtype=torch.bfloat16, device=dev)
    out = torch.empty((1, M, pw_down.N), dtype=torch.bfloat16, device=dev)
    ws_up = torch.empty(ops.workspace_size(1, M, pw_up.N, pw_up.K, False), dtype=torch.uint8, device=dev)
    ws_dn = torch.empty(ops.workspace_size(1, M, pw_down.N, pw_down.K, False), dtype=torch.uint8, device=dev)
    y = ops.PackedActivation(torch.empty((1, M, pw_up.N), dtype=torch.uint8, device=dev),
                             torch.empty(ops.packed_sizes(1, M, pw_up.N)[1], dtype=torch.uint8, device=dev),
                             1, M, pw_up.N)
    lib = ops.load()

    def chain_bf16():
        ops.linear(x, pw_up, out=h, workspace=ws_up)
        ops.linear(h, pw_down, out=out[0], workspace=ws_dn)

    def chain_hand_off():
        ops._check(lib.mxfp8_linear_quantized_out(x.data_ptr(), None, None, 1, M, pw_up.N, pw_up.K,
                                                  pw_up.w_packed.data_ptr(), pw_up.sf_packed.data_ptr(), None,
                                                  None, y.x_q.data_ptr(), y.sf_packed.data_ptr(),
                                                  ws_up.data_ptr(), ws_up.numel(), ops._stream()))
        ops.gemm_packed(y, pw_down, out=out)

    flops = 2.0 * M * pw_up.K * pw_up.N + 2.0 * M * pw_down.K * pw_down.N
    res = {}
    for name, fn in (("bf16_chain", chain_bf16), ("quantized_hand_off", chain_hand_off)):
        us = _time_steps(fn, flush, stream, steps)
        res[name] = {"us": us, "tflops": flops / (us * 1e-6) / 1e12}
    ops.check()
    res["launches"] = {"bf16_chain": 4, "quantized_hand_off": 3}
    return res


ONLY = ("prefill_up", "prefill_down", "bmm", "bmm_fused", "decode_M1", "decode_M16", "decode_M64",
        "chain_hand_off", "medium_M128", "medium_M256", "medium_M512", "up_M128", "quantize_sweep")


def _quantize_sweep(ops, dev, flush, stream, steps):
    """The quantise step (packed scales, as inside mxfp8_linear) over M at
    K = 4096, next to a plain device copy of M x K bytes and a kernel that
    zeroes 256 bytes, all timed the same way (one call between events, L2
    flushed before it; median of `steps`): separates the per-call floor of the
    timing method from the kernel's rate.  One JSON line per size."""
    K = 4096
    g = torch.Generator(device=dev).manual_seed(11)

    def med(fn):
        for _ in range(5):
            fn()
            flush.zero_()
        return statistics.median(_time_calls(fn, flush, stream, steps)) * 1e3

    tiny = torch.empty(256, dtype=torch.uint8, device=dev)
    print(json.dumps({"only": "quantize_sweep", "tiny_kernel_us": med(lambda: tiny.zero_())}), flush=True)
    for M in (2048, 4096, 8192, 16384):
        x = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        x_q = torch.empty((1, M, K), dtype=torch.uint8, device=dev)
        sfa = torch.empty(ops.packed_sizes(1, M, K)[1], dtype=torch.uint8, device=dev)
        src = torch.empty(M * K, dtype=torch.uint8, device=dev)
        dst = torch.empty(M * K, dtype=torch.uint8, device=dev)
        q_us = med(lambda: ops.quantize_packed(x, 1, x_q=x_q, sf_packed=sfa))
        c_us = med(lambda: dst.copy_(src))
        nbytes = 2 * M * K + M * K + M * K // 32
        print(json.dumps({"only": "quantize_sweep", "M": M, "K": K, "bytes": nbytes, "quantize_us": q_us,
                          "copy_MK_bytes_us": c_us}), flush=True)
        del x, x_q, sfa, src, dst
    ops.check()


def run_only(args):
    """--only WORKLOAD: warm-up, then `steps` calls of one workload with the L2
    flushed between calls; prints {"only", "us"}.  For profiling runs (ncu
    launch lists and captures), not the benchmark line."""
    from mxfp8_block_scaled_02_gb300 import build, ops
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    ops.load()
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    w = args.only
    if w == "quantize_sweep":
        _quantize_sweep(ops, dev, flush, stream, args.steps)
        return
    if w.startswith("decode_M") or w.startswith("medium_M"):
        # decode: the first M rows of the decode batch; medium: a prefill chunk
        # of M bf16 rows on the same N = K = 4096 weights (split K over pairs)
        M = int(w.split("_M")[1])
        p = synth.decode(64)
        wq, ws = ops.quantize(_dev_bf16(p.w[0], dev))
        pw = ops.process_weights(wq, ws)
        bias = _dev_bf16(p.bias, dev)
        if w.startswith("decode_M"):
            x = _dev_bf16(p.x[0, :M], dev)
        else:
            x = _dev_bf16(synth.to_bf16_bits(synth.normal(77 + M, M * p.K)).reshape(M, p.K), dev)
        out = torch.empty((M, p.N), dtype=torch.bfloat16, device=dev)
        wsb = torch.empty(max(ops.workspace_size(1, M, p.N, p.K, False), 1), dtype=torch.uint8, device=dev)
        fn = lambda: ops.linear(x, pw, bias, out=out, workspace=wsb, path=args.path)  # noqa: E731
    elif w == "prefill_down":
        p = synth.prefill_down()
        xq, xs = ops.quantize(_dev_bf16(p.x[0], dev))
        wq, ws = ops.quantize(_dev_bf16(p.w[0], dev))
        pw = ops.process_weights(wq, ws)
        out = torch.empty((p.M, p.N), dtype=torch.bfloat16, device=dev)
        wsb = torch.empty(ops.workspace_size(1, p.M, p.N, p.K, True), dtype=torch.uint8, device=dev)
        fn = lambda: ops.linear(xq, pw, x_scale=xs, out=out, workspace=wsb, path=args.path)  # noqa: E731
    else:
        # bmm_fused: the batched workload on the GEMM that quantises x itself (path 5)
        # up_M128: a 128-token chunk (the first 128 rows) through the MLP-up
        # weights: 56 output tiles, so one CTA per 128 x 256 tile, unsplit
        batched = w.startswith("bmm")
        p = synth.bmm() if batched else synth.prefill_up()
        x = _dev_bf16(p.x if batched else p.x[0], dev)
        if w == "up_M128":
            x = x[:128].contiguous()
            p.M = 128
        wq, ws = ops.quantize(_dev_bf16(p.w if batched else p.w[0], dev))
        pw = ops.process_weights(wq, ws)
        out = torch.empty((*x.shape[:-1], p.N), dtype=torch.bfloat16, device=dev)
        wsb = torch.empty(ops.workspace_size(p.B, p.M, p.N, p.K, False), dtype=torch.uint8, device=dev)
        path = 5 if w == "bmm_fused" else args.path
        fn = lambda: ops.linear(x, pw, out=out, workspace=wsb, path=path)  # noqa: E731
        if w == "chain_hand_off":
            r = _two_layer_chain(ops, dev, flush, stream, pw, x, args.steps)
            print(json.dumps({"only": w, **r}), flush=True)
            return
    for _ in range(args.warmup):
        fn()
        flush.zero_()
    ops.check()
    t = _time_calls(fn, flush, stream, args.steps)
    ops.check()
    print(json.dumps({"only": w, "us": statistics.mean(t) * 1e3, "min_us": min(t) * 1e3}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only", choices=ONLY, default=None,
                    help="time one workload alone (for profiling runs; prints no benchmark line)")
    ap.add_argument("--path", type=int, default=0, choices=range(6),
                    help="with --only: the mxfp8_linear_path kernel path (0 = automatic)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.only is not None:
        run_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
