"""Parity of the NVFP4 GEMM (block-scaled FP4 MMA with E4M3 factors,
kind::mxf4nvf4, times the two per-tensor scales) with the oracle:
|C - C_ref| <= 2e-3 * sum_k |a_hat||b_hat| for the fp32 accumulator, plus
half a bf16 ulp for bf16 outputs (the bound of the FP8 GEMM; the products of
E2M1 values and E4M3 factors are exact, so only the accumulation and the
final multiply by gA gB round)."""
import numpy as np
import pytest
import torch

import fgq_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _operands(M, N, K, seed, spread=4):
    a = fgq_inputs.exponent_spread((M, K), spread, 1, seed=seed)
    b = fgq_inputs.exponent_spread((N, K), spread, 1, seed=seed + 1)   # the weight as [N, K]
    aq, sa, ga = oracle.quant_nvfp4_1x16(a)
    bq, sb, gb = oracle.quant_nvfp4_1x16(b)
    return aq, sa, ga, bq, sb, gb


def _dev(host, dev):
    aq, sa, ga, bq, sb, gb = host
    t = lambda v: torch.from_numpy(v).to(dev)
    g = lambda v: torch.tensor([float(v)], dtype=torch.float32, device=dev)
    return t(aq), t(sa), g(ga), t(bq), t(sb), g(gb)


def _check(c_gpu, host, rows=None, cols=None):
    if rows is None:
        cref, tref = oracle.gemm_nvfp4(*host)
        c = c_gpu.float().cpu().numpy().astype(np.float64)
    else:
        cref, tref = oracle.gemm_nvfp4_at(*host, rows, cols)
        c = c_gpu.float().cpu().numpy()[rows, cols].astype(np.float64)
    assert np.isfinite(c).all()
    ok, ratio = oracle.gemm_within_tolerance(c, cref, tref, TOL,
                                             out_bf16=c_gpu.dtype == torch.bfloat16)
    assert ok, f"max |err|/T = {ratio:.3e} exceeds {TOL}"


# (M, N, K): 128-column tiles; K % 256 == 128 leaves a half stage at the end
SHAPES = [(128, 256, 256), (33, 384, 640), (129, 640, 1152), (300, 128, 128), (1000, 512, 1024)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_nvfp4_gemm_narrow_tiles(fgq, cuda_dev, M, N, K, out_dtype):
    host = _operands(M, N, K, seed=M + K)
    c = fgq.gemm_nvfp4(*_dev(host, cuda_dev), out_dtype=out_dtype)
    torch.cuda.synchronize()
    _check(c, host)


@pytest.mark.parametrize("M,K", [(1280, 1024), (1200, 1152)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_nvfp4_gemm_wide_tiles(fgq, cuda_dev, M, K, out_dtype):
    """N = 4096: 128 x 256 tiles; sampled outputs plus every row of the last
    (ragged) tile row."""
    N = 4096
    host = _operands(M, N, K, seed=5)
    c = fgq.gemm_nvfp4(*_dev(host, cuda_dev), out_dtype=out_dtype)
    torch.cuda.synchronize()
    rng = np.random.default_rng(M)
    rows = np.concatenate([rng.integers(0, M, 4000), np.repeat(np.arange(M - 64, M), 4)])
    cols = np.concatenate([rng.integers(0, N, 4000), np.tile([0, 255, 2048, N - 1], 64)])
    _check(c, host, rows, cols)


def _tiles(s, dev):
    """Block scales in the tiled layout, from the oracle's definition."""
    return torch.from_numpy(oracle.fp4_scale_tiles(s)).to(dev)


# Tiled block scales (fgq_gemm_nvfp4_tiled): (M, N, K) over one row tile
# (single CTAs), two or more (CTA pairs on 256- or 128-column tiles), a
# ragged last row tile, an odd number of row tiles (the last pair's second
# CTA has no rows), a final half stage (K % 256 == 128) and K = 128.
TILED_SHAPES = [(128, 256, 256), (33, 384, 640), (129, 640, 1152), (300, 128, 128),
                (1000, 512, 1024), (1100, 5120, 1152), (1280, 4096, 128), (2560, 2048, 2304),
                (640, 7168, 512)]
_TILED_REF = {}


@pytest.mark.parametrize("M,N,K", TILED_SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_nvfp4_gemm_tiled_scales(fgq, cuda_dev, M, N, K, out_dtype):
    """Every output of the first and the last 256 x 256 block (both CTAs'
    rows and both halves of a pair's weight tile), plus sampled outputs."""
    key = (M, N, K)
    if key not in _TILED_REF:  # the reference serves both output types
        host = _operands(M, N, K, seed=M + N)
        m_last = ((M - 1) // 256) * 256
        n_last = max(N - 256, 0)
        blocks = [(r, q) for r0, q0 in ((0, 0), (m_last, n_last))
                  for r in range(r0, min(r0 + 256, M)) for q in range(q0, min(q0 + 256, N))]
        rng = np.random.default_rng(K)
        rows = np.concatenate([np.array([b[0] for b in blocks]), rng.integers(0, M, 3000)])
        cols = np.concatenate([np.array([b[1] for b in blocks]), rng.integers(0, N, 3000)])
        _TILED_REF[key] = (host, rows, cols, oracle.gemm_nvfp4_at(*host, rows, cols))
    host, rows, cols, (cref, tref) = _TILED_REF[key]
    aq, sa, ga, bq, sb, gb = _dev(host, cuda_dev)
    c = fgq.gemm_nvfp4_tiled(aq, _tiles(host[1], cuda_dev), ga, bq, _tiles(host[4], cuda_dev), gb,
                             out_dtype=out_dtype)
    torch.cuda.synchronize()
    c = c.float().cpu().numpy()[rows, cols].astype(np.float64)
    assert np.isfinite(c).all()
    ok, ratio = oracle.gemm_within_tolerance(c, cref, tref, TOL,
                                             out_bf16=out_dtype == torch.bfloat16)
    assert ok, f"max |err|/T = {ratio:.3e} exceeds {TOL}"
    assert fgq.device_error() == 0


def test_nvfp4_gemm_from_the_gpu_quantizer(fgq, cuda_dev):
    """End to end: both operands quantized on the GPU (global scale, then
    blocks; bit-exact with the oracle), then the GEMM."""
    M, N, K = 200, 384, 768
    a = fgq_inputs.normal((M, K), 1.0, seed=8)
    w = fgq_inputs.normal((K, N), 0.02, seed=9)
    aq, sa, ga = fgq.quant_nvfp4_1x16(a.to(cuda_dev))
    bq, sb, gb = fgq.quant_nvfp4_1x16(w.t().contiguous().to(cuda_dev))
    c = fgq.gemm_nvfp4(aq, sa, ga, bq, sb, gb)
    torch.cuda.synchronize()
    host = oracle.quant_nvfp4_1x16(a) + oracle.quant_nvfp4_1x16(w.t().contiguous())
    for gpu, ref in zip((aq, sa, ga, bq, sb, gb), host):
        assert np.array_equal(gpu.cpu().numpy().reshape(np.shape(ref)), ref)
    _check(c, host)
    assert fgq.device_error() == 0


def test_nvfp4_gemm_large_prefill_sampled(fgq, cuda_dev):
    """4096 x 7168 x 7168, bf16 out: sampled outputs."""
    M, N, K = 4096, 7168, 7168
    a, w = fgq_inputs.large_prefill(seed=0)
    host = oracle.quant_nvfp4_1x16(a) + oracle.quant_nvfp4_1x16(w.t().contiguous())
    c = fgq.gemm_nvfp4(*_dev(host, cuda_dev), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    rows = np.concatenate([rng.integers(0, M, 1500), [0, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 1500), [N - 1, 0]])
    _check(c, host, rows, cols)
    assert fgq.device_error() == 0


def test_nvfp4_gemm_tiled_large_prefill_from_the_gpu_quantizer(fgq, cuda_dev):
    """4096 x 7168 x 7168, bf16 out, as the benchmark runs it: both operands
    quantized on the GPU with tiled scales (codes, scales and global scales
    bit for bit the oracle's), then the first 256 x 256 block of C and
    sampled outputs against the oracle."""
    M, N, K = 4096, 7168, 7168
    a, w = fgq_inputs.large_prefill(seed=0)
    wt = w.t().contiguous()
    aq, sa, ga = fgq.quant_nvfp4_1x16_tiled(a.to(cuda_dev))
    bq, sb, gb = fgq.quant_nvfp4_1x16_tiled(wt.to(cuda_dev))
    c = fgq.gemm_nvfp4_tiled(aq, sa, ga, bq, sb, gb, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    host = oracle.quant_nvfp4_1x16(a) + oracle.quant_nvfp4_1x16(wt)
    assert np.array_equal(aq.cpu().numpy(), host[0]) and np.array_equal(bq.cpu().numpy(), host[3])
    assert np.array_equal(sa.cpu().numpy(), oracle.fp4_scale_tiles(host[1]))
    assert np.array_equal(sb.cpu().numpy(), oracle.fp4_scale_tiles(host[4]))
    assert float(ga.cpu()[0]) == float(host[2]) and float(gb.cpu()[0]) == float(host[5])
    rng = np.random.default_rng(1)
    rows = np.concatenate([np.repeat(np.arange(256), 256), rng.integers(0, M, 2000), [M - 1]])
    cols = np.concatenate([np.tile(np.arange(256), 256), rng.integers(0, N, 2000), [N - 1]])
    _check(c, host, rows, cols)
    assert fgq.device_error() == 0


@pytest.mark.parametrize("pair", [False, True], ids=["single", "pair"])
def test_nvfp4_gemm_tiled_padded_c(fgq, cuda_dev, pair):
    """C as rows of a wider buffer (ldc > N, NaN canaries past column N)."""
    M, N, K = (120, 384, 512) if not pair else (600, 2560, 512)
    host = _operands(M, N, K, seed=77 + M)
    aq, sa, ga, bq, sb, gb = _dev(host, cuda_dev)
    buf = torch.full((M, N + 32), float("nan"), dtype=torch.float32, device=cuda_dev)
    c = fgq.gemm_nvfp4_tiled(aq, _tiles(host[1], cuda_dev), ga, bq, _tiles(host[4], cuda_dev), gb,
                             out_dtype=torch.float32, out=buf[:, :N])
    torch.cuda.synchronize()
    assert torch.isnan(buf[:, N:]).all(), "the GEMM wrote past column N"
    _check(c, host)
