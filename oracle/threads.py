"""The oracle's fp64 GEMM reference spread over the host's cores.

TEST INFRASTRUCTURE ONLY, like the rest of this package.  Nothing here does
arithmetic of the method: every value comes from ``oracle.gemm_dequant``
(the dequantised fp64 product and its bound T = sum_k |a_hat| |b_hat|,
"Fine-Grained FP8/FP4 Quantization" page, §DeepGEMM).  This module only
cuts the output into column slices of whole 128x128 weight blocks, runs the
oracle on each slice in a thread (ctypes releases the GIL for the C call),
and writes each slice into its place.  A column slice of C needs only the
matching column blocks of Bq and sB, and each element's sum over k runs in
the same order as in one whole-matrix call, so the result is identical to
``oracle.gemm_dequant`` on the whole matrix, bit for bit.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import gemm_dequant


def default_workers() -> int:
    """Threads to use: the cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def gemm_dequant_parallel(aq, sa, bq, sb, workers: int | None = None, blocks_per_task: int = 1):
    """fp64 (C, T) of the block-scaled GEMM on the whole [M, N] output.

    aq uint8 [M, K], sa float32 [M, K/128], bq uint8 [K, N] (logical layout),
    sb float32 [K/128, N/128].  Tasks are slices of ``blocks_per_task``
    column blocks (128 columns each), run on ``workers`` threads."""
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    bq = np.asarray(bq, dtype=np.uint8)
    sb = np.asarray(sb, dtype=np.float32)
    M, K = aq.shape
    K2, N = bq.shape
    assert K == K2 and N % 128 == 0
    nb = N // 128
    c = np.empty((M, N), dtype=np.float64)
    t = np.empty((M, N), dtype=np.float64)
    workers = workers or default_workers()

    def task(b0):
        b1 = min(nb, b0 + blocks_per_task)
        n0, n1 = 128 * b0, 128 * b1
        cs, ts = gemm_dequant(aq, sa, np.ascontiguousarray(bq[:, n0:n1]),
                              np.ascontiguousarray(sb[:, b0:b1]))
        c[:, n0:n1] = cs
        t[:, n0:n1] = ts

    with ThreadPoolExecutor(max_workers=workers) as pool:
        list(pool.map(task, range(0, nb, blocks_per_task)))
    return c, t
