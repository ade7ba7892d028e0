"""Parity of the 128x1 (transposed) activation quantizer with the oracle.

Groups of 128 consecutive rows of one column of X [M, K], written as the
A operand of a GEMM that reduces over M: codes XqT [K, M] and scales
sXT [K, M/128] (the plainest extension of the 1x128 tiles of
"Fine-Grained FP8/FP4 Quantization", §Scaling Granularities).  Codes and
scales must match the oracle bit for bit; the weight-gradient product
dW = X^T dY computed from them by the block-scaled GEMM must meet the GEMM
bound.
"""
import numpy as np
import pytest
import torch

import fgq_inputs
import oracle

pytestmark = pytest.mark.gpu

MODES = [("fp32", oracle.MODE_FP32), ("ue8m0", oracle.MODE_UE8M0)]


def _check(fgq, x_cpu, mode, dev, ldx_pad=0):
    M, K = x_cpu.shape
    if ldx_pad:
        big = torch.zeros((M, K + ldx_pad), dtype=torch.bfloat16)
        big[:, :K] = x_cpu
        x = big.to(dev)[:, :K]
    else:
        x = x_cpu.to(dev)
    q, s = fgq.quant_act_128x1(x, mode[0])
    torch.cuda.synchronize()
    qo, so = oracle.quant_act_128x1(x_cpu, mode[1])
    qg, sg = q.cpu().numpy(), s.cpu().numpy()
    assert np.array_equal(sg.view(np.uint32), so.view(np.uint32)), "scales differ"
    bad = np.argwhere(qg != qo)
    assert bad.size == 0, f"{len(bad)} codes differ, first at (k, m) = {tuple(bad[0])}"


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
@pytest.mark.parametrize("M,K,pad", [(128, 128, 0), (256, 384, 0), (384, 1024, 64),
                                     (1024, 256, 8)])
def test_128x1_matches_oracle(fgq, cuda_dev, mode, M, K, pad):
    x = fgq_inputs.outlier((M, K), 1e-2, 100.0, seed=M + K)
    _check(fgq, x, mode, cuda_dev, pad)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_128x1_column_scales_across_binades(fgq, cuda_dev, mode):
    """Every column group has its own amax: 1024 columns whose maxima run
    over many binades and significands (including ones below the range of
    the division-free quotient), the other rows random values below it."""
    M, K = 256, 1024
    g = torch.Generator().manual_seed(7)
    e = torch.randint(-120, 60, (K,), generator=g).to(torch.float32)
    sig = 1.0 + torch.randint(0, 128, (K,), generator=g).to(torch.float32) / 128.0
    amax = sig * torch.exp2(e)
    u = torch.rand((M, K), generator=g) * 2.0 - 1.0
    x = (u * amax).to(torch.bfloat16)
    rows = torch.randint(0, 128, (K,), generator=g)
    for mb in range(M // 128):
        x[mb * 128 + rows, torch.arange(K)] = amax.to(torch.bfloat16)
    x[:128, 17] = 0.0                                   # a zero group
    x[128:, 33] = -0.0                                  # a group of negative zeros
    _check(fgq, x, mode, cuda_dev)


def test_128x1_full_size(fgq, cuda_dev):
    """Activations [4096, 7168] Student-t (nu = 3): every code and scale."""
    x = fgq_inputs.student_t((4096, 7168), 3, 1.0, seed=5)
    _check(fgq, x, MODES[0], cuda_dev)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_weight_gradient_gemm_from_128x1(fgq, cuda_dev, mode):
    """dW [K, N] = X^T dY: X [M, K] quantized 128x1 (A operand, reduction over
    M), dY [M, N] quantized 128x128 (B operand); the GEMM of the GPU codes
    meets the bound against the oracle's fp64 product of the same codes."""
    M, K, N = 512, 384, 256
    x = fgq_inputs.normal((M, K), 1.0, seed=11)
    dy = fgq_inputs.normal((M, N), 0.02, seed=12)
    xqt, sxt = fgq.quant_act_128x1(x.to(cuda_dev), mode[0])
    dyq, sdy = fgq.quant_w_128x128(dy.to(cuda_dev), mode[0])
    dw = fgq.gemm_fp8_blockscaled(xqt, sxt, dyq, sdy, out_dtype=torch.float32, mode=mode[0])
    torch.cuda.synchronize()
    aq, sa = oracle.quant_act_128x1(x, mode[1])
    bq, sb = oracle.quant_w_128x128(dy, mode[1])
    assert np.array_equal(xqt.cpu().numpy(), aq) and np.array_equal(dyq.cpu().numpy(), bq.T)
    cref, tref = oracle.gemm_dequant(aq, sa, bq, sb)
    ok, ratio = oracle.gemm_within_tolerance(dw.cpu().numpy().astype(np.float64), cref, tref, 2e-3)
    assert ok, f"max |err|/T = {ratio:.3e}"
    assert fgq.device_error() == 0
