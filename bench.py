"""Benchmark of the fine-grained FP8 hot path on GB300.

One step = the whole hot path on one batch of the large-prefill workload:
  quantize A [4096, 7168] bf16 (1x128 tiles) and B [7168, 7168] bf16 (128x128
  blocks), both in one launch -> block-scaled FP8 GEMM -> C [4096, 7168] bf16.
value = 2*M*N*K / (step time), in TFLOP/s, summed over ranks (weak scaling:
every rank runs its own batch; the path has no exchange step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fgq|reference]

--impl reference times the CPU oracle (the plain C restatement of the
method) on a bounded sample of the same workload on this machine's host
cores, extrapolated to the full step.

Prints one JSON line (rank 0).
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "block-scaled FP8 GEMM TFLOP/s + quantize GB/s, % of GB300 roofline, 1 GPU"
M_, N_, K_ = 4096, 7168, 7168
WORKLOAD = "large_prefill: A bf16 [4096,7168] N(0,1), B bf16 [7168,7168] N(0,0.02^2); " \
           "quantize A 1x128 + B 128x128 (E4M3, fp32 scales), block-scaled FP8 GEMM, bf16 C"

# Algorithmic bytes / flops per launch (one unit = one launch on this workload).
BYTES_QUANT_ACT = M_ * K_ * 2 + M_ * K_ + M_ * (K_ // 128) * 4           # read bf16, write e4m3 + scales
BYTES_QUANT_W = K_ * N_ * 2 + K_ * N_ + (K_ // 128) * (N_ // 128) * 4
FLOPS_GEMM = 2 * M_ * N_ * K_
BYTES_GEMM = M_ * K_ + N_ * K_ + M_ * (K_ // 128) * 4 + (K_ // 128) * (N_ // 128) * 4 + M_ * N_ * 2

SOAK_SECONDS = 1.0  # the sustained leg after the timed region (also the clock record)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """A CUDA source without its comments and blank lines: what the
    compiler sees, so that editing a comment does not retire a capture."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def _kernel_sha(name: str) -> str:
    """First 16 hex digits of the sha256 of the kernel's unit and of
    fgq_device.cuh, comments left out."""
    h = hashlib.sha256()
    for f in (name, "fgq_device.cuh"):
        with open(os.path.join(ROOT, "fine_grained_fp8_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def _traffic(kernel_key: str, source: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since those counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        ent = t[kernel_key]
        if ent.get("source_sha") != _kernel_sha(source):
            return None
        return ent["bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        return None


# ---- clocks -----------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="fgq_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()
        return False

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(rows)}


# ---- distributed plumbing ---------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    dist.init_process_group(backend=backend)
    return dist


def reduce_max(dist, value: float, device) -> float:
    """Max of a per-rank float over all ranks (identity on one rank)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _event_us(fn, stream, n: int) -> float:
    """Mean device time of fn() in microseconds: CUDA events around n calls
    on `stream`, after three untimed ones."""
    import torch
    for _ in range(3):
        fn()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    e1.synchronize()
    return 1e3 * e0.elapsed_time(e1) / n


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---- CPU oracle arm -------------------------------------------------------------

class OracleSample:
    """The oracle on a bounded sample of one step of the workload, on the
    host's cores.

    Setup (untimed) draws the inputs and quantizes the full weight once so the
    GEMM sample has valid operands.  A timed sample quantizes `rows_a`
    activation rows (threads over row slices) and `blocks_w` 128x128 weight
    blocks (threads over blocks), and computes `gemm_rows` whole rows of C
    over the full K (threads over column blocks); each part is scaled
    linearly to the full step.  With workers = 1 everything runs on one
    thread."""

    def __init__(self, seed: int = 0):
        import numpy as np

        import fgq_inputs
        import oracle
        self.np, self.oracle = np, oracle
        self.a, self.b = fgq_inputs.large_prefill(seed=seed)
        self.bq, self.sb = oracle.quant_w_128x128(self.b)

    def step(self, rows_a: int, blocks_w: int, gemm_rows: int, seed: int, workers: int):
        from concurrent.futures import ThreadPoolExecutor

        from oracle.threads import gemm_dequant_parallel
        np, oracle = self.np, self.oracle
        rng = np.random.default_rng(seed)
        r0 = int(rng.integers(0, M_ - rows_a + 1))
        blocks = [(int(rng.integers(0, K_ // 128)) * 128, int(rng.integers(0, N_ // 128)) * 128)
                  for _ in range(blocks_w)]
        parts = max(1, min(workers, rows_a))
        bounds = [r0 + (rows_a * i) // parts for i in range(parts + 1)]
        with ThreadPoolExecutor(max_workers=workers) as pool:
            t0 = time.perf_counter()
            res = list(pool.map(lambda i: oracle.quant_act_1x128(self.a[bounds[i]:bounds[i + 1]]),
                                range(parts)))
            t1 = time.perf_counter()
            list(pool.map(lambda kn: oracle.quant_w_128x128(
                self.b[kn[0]:kn[0] + 128, kn[1]:kn[1] + 128].contiguous()), blocks))
            t2 = time.perf_counter()
        aq = np.concatenate([r[0] for r in res])[:gemm_rows]
        sa = np.concatenate([r[1] for r in res])[:gemm_rows]
        gemm_dequant_parallel(aq, sa, self.bq, self.sb, workers=workers)
        t3 = time.perf_counter()
        full = ((t1 - t0) * (M_ / rows_a) + (t2 - t1) * ((K_ // 128) * (N_ // 128) / blocks_w)
                + (t3 - t2) * (M_ / gemm_rows))
        return full, t3 - t0

    @staticmethod
    def describe(rows_a, blocks_w, gemm_rows, workers):
        return (f"quantize {rows_a}/{M_} activation rows and {blocks_w}/"
                f"{(K_ // 128) * (N_ // 128)} weight blocks, then {gemm_rows}/{M_} whole rows of "
                f"C (all {N_} columns, full K); each part scaled linearly to the full step; "
                f"{workers} thread(s)")


def host_workers() -> int:
    from oracle.threads import default_workers
    return default_workers()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    sampler = OracleSample(seed=0)
    workers = host_workers()
    rows_a, blocks_w, gemm_rows = 256, 4 * workers, 32
    for i in range(args.warmup):
        sampler.step(rows_a, blocks_w, gemm_rows, seed=i, workers=workers)
    fulls, own = [], 0.0
    for i in range(args.steps):
        f, s = sampler.step(rows_a, blocks_w, gemm_rows, seed=1000 + i, workers=workers)
        fulls.append(f)
        own += s
    step_s = sum(fulls) / len(fulls)
    value = FLOPS_GEMM / step_s / 1e12
    sample = "per step: " + OracleSample.describe(rows_a, blocks_w, gemm_rows, workers)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_, "N": N_, "K": K_, "out": "bf16",
                   "scale_mode": "fp32", "parallelism": f"replicas{world}",
                   "sampled_seconds": own},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": workers, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- GPU arm ---------------------------------------------------------------------

def run_fgq(args):
    import torch

    import fgq_inputs
    import fine_grained_fp8_gb300 as fgq
    from fine_grained_fp8_gb300 import build as fbuild

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, os.environ.get("FGQ_BENCH_BACKEND", "nccl"))
    if rank == 0 or not os.path.exists(fbuild.LIB_PATH):
        fbuild.build()
    barrier(dist)
    fgq.load()

    # Two input sets per rank, rotated, so every step reads inputs larger than
    # L2 (A 58.7 MB + B 102.8 MB bf16 per set) that the previous step did not.
    sets = []
    host_sets = []
    for i in range(2):
        a, b = fgq_inputs.large_prefill(seed=100 * rank + 2 * i)
        host_sets.append((a.pin_memory(), b.pin_memory()))
        sets.append((a.to(dev), b.to(dev)))
    aq = torch.empty((M_, K_), dtype=torch.uint8, device=dev)
    sa = torch.empty((M_, K_ // 128), dtype=torch.float32, device=dev)
    bq = torch.empty((N_, K_), dtype=torch.uint8, device=dev)
    sb = torch.empty((K_ // 128, N_ // 128), dtype=torch.float32, device=dev)
    c = torch.empty((M_, N_), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i, ev=None):
        a, b = sets[i % 2]
        if ev is not None:
            ev[0].record(stream)
        fgq.quant_operands(a, b, "fp32", xq=aq, sx=sa, wq=bq, sw=sb)
        if ev is not None:
            ev[1].record(stream)
        fgq.gemm_fp8_blockscaled(aq, sa, bq, sb, torch.bfloat16, "fp32", out=c)
        if ev is not None:
            ev[2].record(stream)

    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for i in range(args.warmup):
        step(i)
    w1.record(stream)
    torch.cuda.synchronize()
    warm_ms = w0.elapsed_time(w1) / args.warmup

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    soak_steps = max(1, int(args.sustained_seconds / max(1e-4, warm_ms * 1e-3)))
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(dist)
        torch.cuda.synchronize()
        # The timed region: K steps back to back with nothing between the
        # kernels (an event recorded between two kernels would cut the
        # programmatic dependent launch that overlaps a kernel's set-up with
        # the previous kernel's tail).
        start.record(stream)
        for i in range(args.steps):
            step(i)
        stop.record(stream)
        # The same K steps again with an event around every kernel, for the
        # per-kernel durations (the roofline of each kernel).
        for i in range(args.steps):
            step(i, events[i])
        # The timed region is a few milliseconds, shorter than one clock
        # sample.  The same steps continue for about a second right after it
        # (timed on their own as the sustained figure), so the sampler, which
        # started before the timed region, also sees the clocks these
        # kernels settle at under the power limit.
        s0.record(stream)
        for i in range(soak_steps):
            step(i)
        s1.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
    clk = clocks.summary()
    sustained_ms = reduce_max(dist, s0.elapsed_time(s1), dev) / soak_steps
    clk["window"] = "from before the timed region to the end of the sustained leg after it"
    ms_total = start.elapsed_time(stop)
    ms_total = reduce_max(dist, ms_total, dev)
    ms_step = ms_total / args.steps
    per = [[e[j].elapsed_time(e[j + 1]) for e in events] for j in range(2)]
    us_quant, us_gemm = (1e3 * sum(p) / len(p) for p in per)
    if fgq.device_error() != 0:
        raise SystemExit("a kernel reported a device wait timeout")

    # e2e: the same step through the public API with host buffers.  Every
    # step copies its inputs from pinned host memory to the device and reads
    # C back into pinned host memory.  The copies run on their own streams,
    # double-buffered, so step i+1's upload and step i-1's download overlap
    # step i's kernels (the order a serving loop would use); events order
    # each buffer's reuse.
    e2e_steps = max(3, min(args.steps, 50))
    c_host = [torch.empty((M_, N_), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    a_dev = [torch.empty((M_, K_), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    b_dev = [torch.empty((K_, N_), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    c_dev = [torch.empty((M_, N_), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    h2d = torch.cuda.Stream(dev)
    d2h = torch.cuda.Stream(dev)

    def e2e_run(n, first=None, last=None):
        uploaded = [None, None]    # inputs of slot j are on the device
        consumed = [None, None]    # the kernels have read slot j's inputs
        computed = [None, None]    # C of slot j is complete
        downloaded = [None, None]  # C of slot j is back on the host
        for i in range(n):
            j = i % 2
            ah, bh = host_sets[i % 2]
            with torch.cuda.stream(h2d):
                if consumed[j] is not None:
                    h2d.wait_event(consumed[j])
                if i == 0 and first is not None:
                    first.record(h2d)
                a_dev[j].copy_(ah, non_blocking=True)
                b_dev[j].copy_(bh, non_blocking=True)
                uploaded[j] = torch.cuda.Event()
                uploaded[j].record(h2d)
            stream.wait_event(uploaded[j])
            if downloaded[j] is not None:
                stream.wait_event(downloaded[j])
            fgq.quant_operands(a_dev[j], b_dev[j], "fp32", xq=aq, sx=sa, wq=bq, sw=sb)
            consumed[j] = torch.cuda.Event()
            consumed[j].record(stream)
            fgq.gemm_fp8_blockscaled(aq, sa, bq, sb, torch.bfloat16, "fp32", out=c_dev[j])
            computed[j] = torch.cuda.Event()
            computed[j].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(computed[j])
                c_host[j].copy_(c_dev[j], non_blocking=True)
                downloaded[j] = torch.cuda.Event()
                downloaded[j].record(d2h)
        if last is not None:
            d2h.wait_event(computed[(n - 1) % 2])
            last.record(d2h)

    e2e_run(3)
    torch.cuda.synchronize()
    barrier(dist)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_run(e2e_steps, e0, e1)
    torch.cuda.synchronize()
    barrier(dist)
    e2e_ms = reduce_max(dist, e0.elapsed_time(e1), dev) / e2e_steps
    del a_dev, b_dev, c_dev, c_host

    # The same step with power-of-two (UE8M0) scales: the quantizers round
    # each scale up to 2^k and the GEMM applies the scales inside the tensor
    # core (block-scaled MMA) instead of promoting every K chunk.
    ue8m0 = None
    if not args.no_ue8m0:
        # Both operands quantized in one launch with the scales written as
        # UE8M0 code tiles, then the code-tile GEMM (CTA pairs, factors
        # loaded by TMA); the scale-writer kernel on fp32 scales is timed
        # beside it for comparison.
        usteps = max(10, min(args.steps, 500))
        uta = torch.empty((fgq.ue8m0_scale_tiles_bytes(M_, K_),), dtype=torch.uint8, device=dev)
        utb = torch.empty((fgq.ue8m0_scale_tiles_bytes(N_, K_),), dtype=torch.uint8, device=dev)

        def ustep(i, ev=None):
            a, b = sets[i % 2]
            if ev is not None:
                ev[0].record(stream)
            fgq.quant_operands_ue8m0_tiles(a, b, xq=aq, sa_tiles=uta, wq=bq, sb_tiles=utb)
            if ev is not None:
                ev[1].record(stream)
            fgq.gemm_fp8_ue8m0_tiled(aq, uta, bq, utb, torch.bfloat16, out=c)
            if ev is not None:
                ev[2].record(stream)

        uev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(usteps)]
        for i in range(5):
            ustep(i, uev[i])
        torch.cuda.synchronize()
        u0 = torch.cuda.Event(enable_timing=True)
        u1 = torch.cuda.Event(enable_timing=True)
        u0.record(stream)
        for i in range(usteps):
            ustep(i)
        u1.record(stream)
        for i in range(usteps):
            ustep(i, uev[i])
        torch.cuda.synchronize()
        ums = reduce_max(dist, u0.elapsed_time(u1), dev) / usteps
        uper = [[e[j].elapsed_time(e[j + 1]) for e in uev] for j in range(2)]
        u_quant, u_gemm = (1e3 * sum(p) / len(p) for p in uper)
        fgq.quant_operands(sets[0][0], sets[0][1], "ue8m0", xq=aq, sx=sa, wq=bq, sw=sb)
        u_ex = _event_us(lambda: fgq.gemm_fp8_blockscaled(aq, sa, bq, sb, torch.bfloat16, "ue8m0",
                                                          out=c), stream, 20)
        ue8m0 = {"scale_mode": "ue8m0", "steps": usteps, "ms_per_step": ums,
                 "value": world * FLOPS_GEMM / (ums * 1e-3) / 1e12, "unit": "TFLOP/s",
                 "quant_operands_us": u_quant, "gemm_us": u_gemm,
                 "gemm_TFLOP/s": FLOPS_GEMM / (u_gemm * 1e-6) / 1e12,
                 "gemm_scale_writers_us": u_ex,
                 "kernel": "gemm_fp4_tiled_kernel<pair, 256, MXF8> (tcgen05.mma.cta_group::2 "
                           "kind::mxf8f6f4.block_scale, UE8M0 code tiles by TMA)"}
        del uta, utb
        if fgq.device_error() != 0:
            raise SystemExit("a kernel reported a device wait timeout")

    # MXFP4 on the same workload: A quantized (E2M1, UE8M0 per 32) every step,
    # the weight quantized once as its transpose [N, K] (inference), and the
    # block-scaled FP4 GEMM (tcgen05.mma kind::mxf4), with the block scales
    # in the tiled layout (written so by the quantizer, loaded by TMA).
    mxfp4 = None
    if not args.no_mxfp4:
        msteps = max(10, min(args.steps, 500))
        wq4 = [fgq.quant_mxfp4_1x32_tiled(b.t().contiguous()) for _, b in sets]
        aq4 = torch.empty((M_, K_ // 2), dtype=torch.uint8, device=dev)
        sa4 = torch.empty((fgq.fp4_scale_tiles_bytes(M_, K_ // 32),), dtype=torch.uint8, device=dev)

        def mstep(i, ev=None):
            a, _ = sets[i % 2]
            if ev is not None:
                ev[0].record(stream)
            fgq.quant_mxfp4_1x32_tiled(a, xq=aq4, s_tiles=sa4)
            if ev is not None:
                ev[1].record(stream)
            fgq.gemm_mxfp4_tiled(aq4, sa4, *wq4[i % 2], torch.bfloat16, out=c)
            if ev is not None:
                ev[2].record(stream)

        mev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(msteps)]
        for i in range(5):
            mstep(i, mev[i])
        torch.cuda.synchronize()
        m0 = torch.cuda.Event(enable_timing=True)
        m1 = torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        for i in range(msteps):
            mstep(i)
        m1.record(stream)
        for i in range(msteps):
            mstep(i, mev[i])
        torch.cuda.synchronize()
        mms = reduce_max(dist, m0.elapsed_time(m1), dev) / msteps
        m_act = 1e3 * sum(e[0].elapsed_time(e[1]) for e in mev) / msteps
        m_gemm = 1e3 * sum(e[1].elapsed_time(e[2]) for e in mev) / msteps
        # the same GEMM on row-major scales (factor-writer warps), for comparison
        sa4r = fgq.quant_mxfp4_1x32(sets[0][0])
        wq4r = fgq.quant_mxfp4_1x32(sets[0][1].t().contiguous())
        m_rm = _event_us(lambda: fgq.gemm_mxfp4(*sa4r, *wq4r, torch.bfloat16, out=c), stream, 20)
        mxfp4 = {"format": "MXFP4 (E2M1, UE8M0 scale per 32, both operands along K; "
                           "block scales in the tiled layout)",
                 "steps": msteps, "ms_per_step": mms,
                 "value": world * FLOPS_GEMM / (mms * 1e-3) / 1e12, "unit": "TFLOP/s",
                 "quant_act_us": m_act, "gemm_us": m_gemm,
                 "gemm_TFLOP/s": FLOPS_GEMM / (m_gemm * 1e-6) / 1e12,
                 "gemm_rowmajor_scales_us": m_rm,
                 "kernel": "gemm_fp4_tiled_kernel<pair, 256> (tcgen05.mma.cta_group::2 "
                           "kind::mxf4.block_scale)"}
        del wq4, aq4, sa4, sa4r, wq4r
        if fgq.device_error() != 0:
            raise SystemExit("a kernel reported a device wait timeout")

    # NVFP4 on the same workload: A's per-tensor scale and its E2M1 codes with
    # an E4M3 scale per 16 every step, the weight quantized once as its
    # transpose, and the block-scaled FP4 GEMM with E4M3 factors
    # (tcgen05.mma kind::mxf4nvf4) times the two per-tensor scales.
    nvfp4 = None
    if not args.no_nvfp4:
        nsteps = max(10, min(args.steps, 500))
        wn4 = [fgq.quant_nvfp4_1x16_tiled(b.t().contiguous()) for _, b in sets]
        an4 = torch.empty((M_, K_ // 2), dtype=torch.uint8, device=dev)
        sn4 = torch.empty((fgq.fp4_scale_tiles_bytes(M_, K_ // 16),), dtype=torch.uint8, device=dev)
        gn4 = torch.empty((1,), dtype=torch.float32, device=dev)

        def nstep(i, ev=None):
            a, _ = sets[i % 2]
            if ev is not None:
                ev[0].record(stream)
            fgq.nvfp4_global_scale(a, g=gn4)
            fgq.quant_nvfp4_1x16_tiled(a, g=gn4, xq=an4, s_tiles=sn4)
            if ev is not None:
                ev[1].record(stream)
            bq4, bs4, bg4 = wn4[i % 2]
            fgq.gemm_nvfp4_tiled(an4, sn4, gn4, bq4, bs4, bg4, torch.bfloat16, out=c)
            if ev is not None:
                ev[2].record(stream)

        nev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nsteps)]
        for i in range(5):
            nstep(i, nev[i])
        torch.cuda.synchronize()
        n0 = torch.cuda.Event(enable_timing=True)
        n1 = torch.cuda.Event(enable_timing=True)
        n0.record(stream)
        for i in range(nsteps):
            nstep(i)
        n1.record(stream)
        for i in range(nsteps):
            nstep(i, nev[i])
        torch.cuda.synchronize()
        nms = reduce_max(dist, n0.elapsed_time(n1), dev) / nsteps
        n_act = 1e3 * sum(e[0].elapsed_time(e[1]) for e in nev) / nsteps
        n_gemm = 1e3 * sum(e[1].elapsed_time(e[2]) for e in nev) / nsteps
        an4r = fgq.quant_nvfp4_1x16(sets[0][0])
        wn4r = fgq.quant_nvfp4_1x16(sets[0][1].t().contiguous())
        n_rm = _event_us(lambda: fgq.gemm_nvfp4(*an4r, *wn4r, torch.bfloat16, out=c), stream, 20)
        nvfp4 = {"format": "NVFP4 (E2M1, E4M3 scale per 16 and an fp32 per-tensor scale, "
                           "both operands along K; block scales in the tiled layout)",
                 "steps": nsteps, "ms_per_step": nms,
                 "value": world * FLOPS_GEMM / (nms * 1e-3) / 1e12, "unit": "TFLOP/s",
                 "quant_act_us": n_act, "gemm_us": n_gemm,
                 "gemm_TFLOP/s": FLOPS_GEMM / (n_gemm * 1e-6) / 1e12,
                 "gemm_rowmajor_scales_us": n_rm,
                 "kernel": "gemm_fp4_tiled_kernel<pair, 256, NV> (tcgen05.mma.cta_group::2 "
                           "kind::mxf4nvf4.block_scale.scale_vec::4X)"}
        del wn4, an4, sn4, gn4, an4r, wn4r
        if fgq.device_error() != 0:
            raise SystemExit("a kernel reported a device wait timeout")

    # The quantizers on the quantize-bandwidth workload (activations
    # [16384, 7168] Student-t nu=3, weight [7168, 7168] N(0, 0.02^2)), each
    # timed alone over rotated input pairs larger than L2.
    quant_bw = None
    if not args.no_quant_bw:
        del sets, host_sets
        torch.cuda.empty_cache()
        qa = [fgq_inputs.quant_bw(seed=100 * rank + 2 * i)[0].to(dev) for i in range(2)]
        qw = [fgq_inputs.quant_bw(seed=100 * rank + 2 * i, m=128)[1].to(dev) for i in range(2)]
        QM, QK = qa[0].shape
        qaq = torch.empty((QM, QK), dtype=torch.uint8, device=dev)
        qsa = torch.empty((QM, QK // 128), dtype=torch.float32, device=dev)
        quant_bw = {"workload": "quantize-bw: act bf16 [16384,7168] Student-t nu=3 (1x128, 128x1 "
                                "transposed, MXFP4 1x32, NVFP4 per-tensor scale and 1x16); weight "
                                "bf16 [7168,7168] N(0,0.02^2) (128x128); fp32 scales"}
        qsteps = max(10, min(args.steps, 200))
        qaqt = torch.empty((QK, QM), dtype=torch.uint8, device=dev)
        qmx = torch.empty((QM, QK // 2), dtype=torch.uint8, device=dev)
        qmxs = torch.empty((QM, QK // 32), dtype=torch.uint8, device=dev)
        qsat = torch.empty((QK, QM // 128), dtype=torch.float32, device=dev)
        qnv = torch.empty((QM, QK // 2), dtype=torch.uint8, device=dev)
        qnvs = torch.empty((QM, QK // 16), dtype=torch.uint8, device=dev)
        qmxt = torch.empty((fgq.fp4_scale_tiles_bytes(QM, QK // 32),), dtype=torch.uint8, device=dev)
        qnvt = torch.empty((fgq.fp4_scale_tiles_bytes(QM, QK // 16),), dtype=torch.uint8, device=dev)
        qg = [fgq.nvfp4_global_scale(qa[i]) for i in range(2)]
        qg_out = torch.empty((1,), dtype=torch.float32, device=dev)
        for name, fn, nbytes in (
                ("quant_act_1x128", lambda i: fgq.quant_act_1x128(qa[i % 2], "fp32", xq=qaq, sx=qsa),
                 QM * QK * 3 + QM * (QK // 128) * 4),
                ("quant_act_128x1", lambda i: fgq.quant_act_128x1(qa[i % 2], "fp32", xqt=qaqt, sxt=qsat),
                 QM * QK * 3 + QK * (QM // 128) * 4),
                ("quant_mxfp4_1x32", lambda i: fgq.quant_mxfp4_1x32(qa[i % 2], xq=qmx, sx=qmxs),
                 QM * QK * 2 + QM * QK // 2 + QM * (QK // 32)),
                ("quant_mxfp4_1x32_tiled",
                 lambda i: fgq.quant_mxfp4_1x32_tiled(qa[i % 2], xq=qmx, s_tiles=qmxt),
                 QM * QK * 2 + QM * QK // 2 + QM * (QK // 32)),
                ("nvfp4_global_scale", lambda i: fgq.nvfp4_global_scale(qa[i % 2], g=qg_out),
                 QM * QK * 2 + 4),
                ("quant_nvfp4_1x16", lambda i: fgq.quant_nvfp4_1x16(qa[i % 2], g=qg[i % 2], xq=qnv,
                                                                    sx=qnvs),
                 QM * QK * 2 + QM * QK // 2 + QM * (QK // 16)),
                ("quant_nvfp4_1x16_tiled",
                 lambda i: fgq.quant_nvfp4_1x16_tiled(qa[i % 2], g=qg[i % 2], xq=qnv, s_tiles=qnvt),
                 QM * QK * 2 + QM * QK // 2 + QM * (QK // 16)),
                ("quant_w_128x128", lambda i: fgq.quant_w_128x128(qw[i % 2], "fp32", wq=bq, sw=sb),
                 BYTES_QUANT_W),
                ("quant_operands", lambda i: fgq.quant_operands(qa[i % 2], qw[i % 2], "fp32", xq=qaq,
                                                                sx=qsa, wq=bq, sw=sb),
                 QM * QK * 3 + QM * (QK // 128) * 4 + BYTES_QUANT_W)):
            for i in range(5):
                fn(i)
            torch.cuda.synchronize()
            q0 = torch.cuda.Event(enable_timing=True)
            q1 = torch.cuda.Event(enable_timing=True)
            q0.record(stream)
            for i in range(qsteps):
                fn(i)
            q1.record(stream)
            torch.cuda.synchronize()
            us = reduce_max(dist, q0.elapsed_time(q1), dev) * 1e3 / qsteps
            gbs = nbytes / (us * 1e-6) / 1e9
            quant_bw[name] = {"us": us, "GB/s": gbs, "bytes": nbytes, "launches": qsteps}
        if fgq.device_error() != 0:
            raise SystemExit("a kernel reported a device wait timeout")

    # The skinny sweep (M in {16, 64, 256} x N = 24576 x K = 1536, bf16 out):
    # the low-M GEMM paths, bound by streaming the 37.7 MB of weight codes.
    # Four weight copies (151 MB, more than L2) are rotated, and the launches
    # are replayed from a CUDA graph so host launch time does not count.
    skinny = None
    if not args.no_skinny:
        SN, SK = 24576, 1536
        skinny = {"workload": "skinny: M x N=24576 x K=1536, A N(0,1), B N(0,0.02^2), bf16 out; "
                              "4 weight copies rotated (151 MB > L2); CUDA-graph replay"}
        wcopies = []
        for i in range(4):
            bsk = fgq_inputs.skinny(16, seed=10 + i)[1].to(dev)
            wcopies.append(fgq.quant_w_128x128(bsk))
            del bsk
        for Ms in (16, 64, 256):
            ask = fgq_inputs.skinny(Ms, seed=Ms)[0].to(dev)
            aqs, sas = fgq.quant_act_1x128(ask)
            cs = torch.empty((Ms, SN), dtype=torch.bfloat16, device=dev)
            ws = fgq.splitk_workspace(Ms, SN, SK, dev)
            entry = {}
            timed = [
                ("gemm_fp8_blockscaled", lambda j: fgq.gemm_fp8_blockscaled(
                    aqs, sas, *wcopies[j % 4], torch.bfloat16, out=cs)),
                ("gemm_fp8_blockscaled_splitk", lambda j: fgq.gemm_fp8_blockscaled_splitk(
                    aqs, sas, *wcopies[j % 4], ws, torch.bfloat16, out=cs))]
            if Ms <= 32:
                # bf16 activations in: quantizer then GEMM (two launches) against
                # the GEMM that quantizes A itself (one launch)
                timed += [
                    ("quant_act_then_gemm", lambda j: (
                        fgq.quant_act_1x128(ask, xq=aqs, sx=sas),
                        fgq.gemm_fp8_blockscaled(aqs, sas, *wcopies[j % 4], torch.bfloat16, out=cs))),
                    ("gemm_fp8_blockscaled_fused_act", lambda j: fgq.gemm_fp8_blockscaled_fused_act(
                        ask, *wcopies[j % 4], torch.bfloat16, out=cs))]
            for name, fn in timed:
                for j in range(8):
                    fn(j)
                torch.cuda.synchronize()
                reps = 40
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for j in range(reps):
                        fn(j)
                g.replay()
                torch.cuda.synchronize()
                g0 = torch.cuda.Event(enable_timing=True)
                g1 = torch.cuda.Event(enable_timing=True)
                g0.record(stream)
                for _ in range(5):
                    g.replay()
                g1.record(stream)
                torch.cuda.synchronize()
                us = reduce_max(dist, g0.elapsed_time(g1), dev) * 1e3 / (5 * reps)
                entry[name] = {"us": us}
            nbytes = SN * SK + Ms * SK + Ms * SN * 2 + Ms * (SK // 128) * 4 + (SK // 128) * (SN // 128) * 4
            for name in entry:
                us = entry[name]["us"]
                entry[name]["GB/s"] = nbytes / (us * 1e-6) / 1e9
                entry[name]["TFLOP/s"] = 2 * Ms * SN * SK / (us * 1e-6) / 1e12
            skinny[f"M{Ms}"] = {"bytes": nbytes, "flops": 2 * Ms * SN * SK, **entry}
            del ask, aqs, sas, cs, ws
        del wcopies
        if fgq.device_error() != 0:
            raise SystemExit("a kernel reported a device wait timeout")

    # CPU baseline: the oracle on a bounded sample, rank 0 only, N = 1 only,
    # on all of the host's cores (and, beside it, on one thread).
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sampler = OracleSample(seed=0)
        workers = host_workers()
        full_s, took = sampler.step(M_, (K_ // 128) * (N_ // 128), 256, seed=0, workers=workers)
        one_s, one_took = sampler.step(256, 64, 4, seed=1, workers=1)
        cpu = {"value": FLOPS_GEMM / full_s / 1e12, "unit": "TFLOP/s", "cores": workers,
               "kind": "oracle",
               "sample": OracleSample.describe(M_, (K_ // 128) * (N_ // 128), 256, workers)
                         + f"; {took:.1f} s wall",
               "full_step_s": full_s,
               "single_thread": {"value": FLOPS_GEMM / one_s / 1e12, "unit": "TFLOP/s",
                                 "full_step_s": one_s,
                                 "sample": OracleSample.describe(256, 64, 4, 1)
                                           + f"; {one_took:.1f} s"}}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, src = _peaks()
    if quant_bw:
        for k in ("quant_act_1x128", "quant_act_128x1", "quant_mxfp4_1x32",
                  "quant_mxfp4_1x32_tiled", "nvfp4_global_scale", "quant_nvfp4_1x16",
                  "quant_nvfp4_1x16_tiled", "quant_w_128x128", "quant_operands"):
            quant_bw[k]["frac_hbm"] = quant_bw[k]["GB/s"] / peaks["hbm_gbs"]
    if skinny:
        for k, v in skinny.items():
            if isinstance(v, dict):
                for e in v.values():
                    if isinstance(e, dict):
                        e["frac_hbm"] = e["GB/s"] / peaks["hbm_gbs"]
    # Every GEMM here is timed over a sub-second region, so its denominator is
    # the burst peak: dense fp8 = 2 x the measured bf16 burst (nominal 4.5 /
    # 2.25 PFLOP/s), fp4 = 6 x (nominal 13.5 / 2.25).  The sustained figure
    # is reported beside it.
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    fp8_peak_sustained = 2.0 * peaks["bf16_tflops_sustained"]
    if mxfp4:
        fp4_peak = 6.0 * peaks["bf16_tflops"]  # nominal fp4 = 6x bf16 dense on GB300
        mxfp4["peak_fp4"] = fp4_peak
        mxfp4["frac_fp4"] = mxfp4["gemm_TFLOP/s"] / fp4_peak
        mxfp4["peak_source"] = f"{src}: 6 x bf16_tflops (burst; nominal 13.5 / 2.25 PFLOP/s)"
        mxfp4["traffic"] = _traffic("gemm_mxf4_tiled", "gemm_mxf4.cu")
    if nvfp4:
        fp4_peak = 6.0 * peaks["bf16_tflops"]
        nvfp4["peak_fp4"] = fp4_peak
        nvfp4["frac_fp4"] = nvfp4["gemm_TFLOP/s"] / fp4_peak
        nvfp4["peak_source"] = f"{src}: 6 x bf16_tflops (burst; nominal 13.5 / 2.25 PFLOP/s)"
        nvfp4["traffic"] = _traffic("gemm_nvf4_tiled", "gemm_mxf4.cu")
    if ue8m0:
        ue8m0["frac_fp8"] = ue8m0["gemm_TFLOP/s"] / fp8_peak
        ue8m0["peak_fp8"] = fp8_peak
        ue8m0["traffic"] = _traffic("gemm_mx8_tiled", "gemm_mxf4.cu")
    if skinny and "M16" in skinny:
        skinny["M16"]["traffic_lowm"] = _traffic("gemm_lowm_m16", "gemm_lowm.cu")
    hbm = peaks["hbm_gbs"]
    # The quantizers' half of the metric: each HBM-bound quantizer timed alone
    # on the quantize-bandwidth workload, and the two inside the step.
    quant_roofline = []
    if quant_bw:
        for k in ("quant_act_1x128", "quant_w_128x128", "quant_operands", "quant_act_128x1",
                  "quant_mxfp4_1x32", "quant_mxfp4_1x32_tiled", "nvfp4_global_scale",
                  "quant_nvfp4_1x16", "quant_nvfp4_1x16_tiled"):
            quant_roofline.append({"kernel": k, "workload": "quantize-bw (alone)", "bound": "hbm",
                                   "achieved": quant_bw[k]["GB/s"], "peak": hbm, "unit": "GB/s",
                                   "frac": quant_bw[k]["GB/s"] / hbm,
                                   "bytes_per_launch": quant_bw[k]["bytes"]})
    gemm_tflops = FLOPS_GEMM / (us_gemm * 1e-6) / 1e12
    quant_gbs = (BYTES_QUANT_ACT + BYTES_QUANT_W) / (us_quant * 1e-6) / 1e9
    value = world * FLOPS_GEMM / (ms_step * 1e-3) / 1e12
    for k, us, nbytes in (("quant_operands", us_quant, BYTES_QUANT_ACT + BYTES_QUANT_W),):
        gbs = nbytes / (us * 1e-6) / 1e9
        quant_roofline.append({"kernel": k, "workload": "large prefill (inside the step)",
                               "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                               "frac": gbs / hbm, "bytes_per_launch": nbytes})
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_, "N": N_, "K": K_, "out": "bf16",
                   "scale_mode": "fp32", "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (two input sets rotated, 161 MB bf16 each)",
                   "value_def": "2*M*N*K per step / step time (quantize A and B in one launch + GEMM)"},
        "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": gemm_tflops / fp8_peak,
                     "traffic": _traffic("gemm_fp8_blockscaled", "gemm.cu"),
                     "kernel": "gemm_fp8_blockscaled_kernel",
                     "peak_source": f"{src}: 2 x bf16_tflops (burst; fp8 = 2x bf16 nominal)",
                     "frac_of_sustained": gemm_tflops / fp8_peak_sustained,
                     "quantizers": quant_roofline},
        "kernels": {
            "quant_operands": {"us": us_quant, "GB/s": quant_gbs, "frac_hbm": quant_gbs / hbm,
                               "bytes": BYTES_QUANT_ACT + BYTES_QUANT_W,
                               "what": "quantize A 1x128 and B 128x128 in one launch"},
            "gemm_fp8_blockscaled": {"us": us_gemm, "TFLOP/s": gemm_tflops,
                                     "frac_fp8": gemm_tflops / fp8_peak, "flops": FLOPS_GEMM},
            "fp8_peak": fp8_peak, "fp8_peak_sustained": fp8_peak_sustained,
            "hbm_peak_gbs": hbm, "peak_source": src,
        },
        "e2e": {"value": world * FLOPS_GEMM / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": (M_ * K_ + K_ * N_) * 2, "d2h_bytes_per_step": M_ * N_ * 2,
                "ms_per_step": e2e_ms, "steps": e2e_steps},
        "sustained": {"steps": soak_steps, "ms_per_step": sustained_ms,
                      "value": world * FLOPS_GEMM / (sustained_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                      "note": "the same step repeated for about a second right after the timed "
                              "region (clocks settle under the power limit)"},
        "gpu_launches": 2 * args.steps,
        "quant_bw": quant_bw,
        "ue8m0": ue8m0,
        "mxfp4": mxfp4,
        "nvfp4": nvfp4,
        "skinny": skinny,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["fgq", "reference"], default="fgq")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--sustained-seconds", type=float, default=SOAK_SECONDS,
                   help="length of the sustained leg after the timed region (at least one step)")
    p.add_argument("--no-quant-bw", action="store_true",
                   help="skip the separate quantize-bandwidth measurement")
    p.add_argument("--no-ue8m0", action="store_true",
                   help="skip the power-of-two scale (UE8M0) step")
    p.add_argument("--no-skinny", action="store_true",
                   help="skip the skinny-GEMM sweep")
    p.add_argument("--no-mxfp4", action="store_true",
                   help="skip the MXFP4 step")
    p.add_argument("--no-nvfp4", action="store_true",
                   help="skip the NVFP4 step")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_fgq(args)


if __name__ == "__main__":
    sys.exit(main())
