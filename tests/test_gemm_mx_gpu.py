"""Parity of the GEMM's power-of-two scale path with the oracle.

In UE8M0 mode the scales are applied by the tensor core itself (block-scaled
MMA with the codes in TMEM; "Fine-Grained FP8/FP4 Quantization",
§Blackwell: Native Block Scaling), not by promoting per-chunk partials.
The bar is the one every GEMM test uses (§DeepGEMM):
|C - C_ref| <= 2e-3 * sum_k |a_hat||b_hat| for the fp32 accumulator, plus
half a bf16 ulp for bf16 outputs.  The cases cover both tile widths (128
and 256 columns), K chunk counts that leave a partial group of four in the
scale-factor ring, ragged M, scales spread over many binades, and the
smallest code (2^-127).
"""
import numpy as np
import pytest
import torch

import fgq_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = 2e-3
UE8M0 = oracle.MODE_UE8M0


def _quant(a, b, mode=UE8M0):
    aq, sa = oracle.quant_act_1x128(a, mode)
    bq, sb = oracle.quant_w_128x128(b, mode)
    return aq, sa, bq, sb


def _dev(aq, sa, bq, sb, dev):
    return (torch.from_numpy(aq).to(dev), torch.from_numpy(sa).to(dev),
            torch.from_numpy(np.ascontiguousarray(bq.T)).to(dev), torch.from_numpy(sb).to(dev))


def _check(c_gpu, host, rows=None, cols=None):
    if rows is None:
        cref, tref = oracle.gemm_dequant(*host)
        c = c_gpu.float().cpu().numpy().astype(np.float64)
    else:
        cref, tref = oracle.gemm_dequant_at(*host, rows, cols)
        c = c_gpu.float().cpu().numpy()[rows, cols].astype(np.float64)
    assert np.isfinite(c).all()
    ok, ratio = oracle.gemm_within_tolerance(c, cref, tref, TOL,
                                             out_bf16=c_gpu.dtype == torch.bfloat16)
    assert ok, f"max |err|/T = {ratio:.3e} exceeds {TOL}"
    return ratio


# (M, N, K): 128-column tiles (too few 256-wide tiles, or N % 256 != 0);
# 1, 5, 9 and 18 chunks (partial last group of the four-chunk slots, and
# several passes around the four-slot ring)
SHAPES = [(33, 384, 640), (128, 256, 128), (129, 640, 1152), (300, 128, 2304),
          (1000, 512, 1024)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_ue8m0_narrow_tiles(fgq, cuda_dev, M, N, K, out_dtype):
    a = fgq_inputs.exponent_spread((M, K), 20, 1, seed=M)
    b = fgq_inputs.exponent_spread((K, N), 20, 128, seed=M + 1)
    host = _quant(a, b)
    c = fgq.gemm_fp8_blockscaled(*_dev(*host, cuda_dev), out_dtype=out_dtype, mode="ue8m0")
    torch.cuda.synchronize()
    _check(c, host)


@pytest.mark.parametrize("M,N,K", [(1280, 4096, 640), (1200, 4096, 1152), (1100, 4096, 640),
                                   (384, 8192, 512)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_ue8m0_large_n(fgq, cuda_dev, M, N, K, out_dtype):
    """M = 1280 and 1200 with N = 4096 give at least one 128 x 256 tile per
    SM (one accumulator; the next tile waits for the epilogue's read), the
    last one ragged for M = 1200; M = 1100 and 384 fall back to 128 x 128
    tiles with a ragged last tile row."""
    a = fgq_inputs.exponent_spread((M, K), 12, 1, seed=7)
    b = fgq_inputs.exponent_spread((K, N), 12, 128, seed=8)
    host = _quant(a, b)
    c = fgq.gemm_fp8_blockscaled(*_dev(*host, cuda_dev), out_dtype=out_dtype, mode="ue8m0")
    torch.cuda.synchronize()
    rng = np.random.default_rng(M)
    rows = np.concatenate([rng.integers(0, M, 4000), np.arange(M - 8, M), [0]])
    cols = np.concatenate([rng.integers(0, N, 4000), np.arange(N - 8, N), [0]])
    _check(c, host, rows, cols)
    # every row of the last (ragged) tile row and every column block
    r2 = np.repeat(np.arange(M - 64, M), N // 128)
    c2 = np.tile(np.arange(0, N, 128) + 127, 64)
    _check(c, host, r2, c2)


def test_ue8m0_matches_the_promotion_path(fgq, cuda_dev):
    """Power-of-two scales also go through the fp32-scale (promotion)
    kernel: both results lie within the bound of the oracle."""
    M, N, K = 520, 768, 1536
    a = fgq_inputs.exponent_spread((M, K), 10, 1, seed=11)
    b = fgq_inputs.exponent_spread((K, N), 10, 128, seed=12)
    host = _quant(a, b)
    ops = _dev(*host, cuda_dev)
    c_mx = fgq.gemm_fp8_blockscaled(*ops, out_dtype=torch.float32, mode="ue8m0")
    c_pr = fgq.gemm_fp8_blockscaled(*ops, out_dtype=torch.float32, mode="fp32")
    torch.cuda.synchronize()
    _check(c_mx, host)
    _check(c_pr, host)


def test_ue8m0_extreme_codes(fgq, cuda_dev):
    """Rows whose scales clamp at the smallest code (2^-127), all-zero rows
    (scale 1), and rows 2^30 larger, against weights scaled by 2^40: every
    product stays a normal fp32 number, so the bound holds for each row."""
    M, N, K = 256, 384, 512
    a = fgq_inputs.normal((M, K), 1.0, seed=21).float()
    rowf = torch.ones(M)
    rowf[0:32] = 2.0 ** -122     # amax/448 below 2^-127 (amax < 14): code 0
    rowf[32:40] = 0.0            # zero groups: scale 1 (code 127)
    rowf[40:72] = 2.0 ** 30
    a = (a * rowf[:, None]).to(torch.bfloat16)
    b = (fgq_inputs.normal((K, N), 0.02, seed=22).float() * 2.0 ** 40).to(torch.bfloat16)
    host = _quant(a, b)
    assert (host[1][0:32] == 2.0 ** -127).all(), "the tiny rows should take the smallest code"
    c = fgq.gemm_fp8_blockscaled(*_dev(*host, cuda_dev), out_dtype=torch.float32, mode="ue8m0")
    torch.cuda.synchronize()
    _check(c, host)
    assert (c[32:40] == 0).all()


def test_ue8m0_repeat_calls_are_identical(fgq, cuda_dev):
    M, N, K = 700, 1024, 2048
    a = fgq_inputs.exponent_spread((M, K), 8, 1, seed=31)
    b = fgq_inputs.exponent_spread((K, N), 8, 128, seed=32)
    ops = _dev(*_quant(a, b), cuda_dev)
    c1 = fgq.gemm_fp8_blockscaled(*ops, out_dtype=torch.bfloat16, mode="ue8m0")
    c2 = fgq.gemm_fp8_blockscaled(*ops, out_dtype=torch.bfloat16, mode="ue8m0")
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


def test_no_device_error_after_ue8m0(fgq, cuda_dev):
    assert fgq.device_error() == 0


# ---- UE8M0 code tiles (fgq_gemm_fp8_ue8m0_tiled) ---------------------------------

def _code_tiles(codes):
    """UE8M0 codes [R, F] in the tiled layout: the FP4 scale tiles of the
    oracle with F padded to a multiple of 4 (padding codes 0)."""
    R, F = codes.shape
    F4 = -(-F // 4) * 4
    pad = np.zeros((R, F4), dtype=np.uint8)
    pad[:, :F] = codes
    return oracle.fp4_scale_tiles(pad)


def _codes(s):
    return np.vectorize(oracle.ue8m0_code, otypes=[np.uint8])(s.astype(np.float64))


def _host_tiles(host):
    """Activation code tiles (row m: codes of sA[m, :]) and weight code tiles
    (row n: codes of sB[:, n / 128]) from the oracle's scales."""
    aq, sa, bq, sb = host
    N = bq.shape[1]
    ta = _code_tiles(_codes(sa))
    tb = _code_tiles(_codes(np.repeat(sb, 128, axis=1)[:, :N].T))
    return ta, tb


def _defined(R, K):
    F = K // 128
    F4 = -(-F // 4) * 4
    m = np.zeros((R, F4), dtype=np.uint8)
    m[:, :F] = 1
    return oracle.fp4_scale_tiles(m) == 1


@pytest.mark.parametrize("M,N,K", [(33, 384, 640), (300, 1024, 1536), (4096, 512, 7168)])
def test_ue8m0_scale_tiles_match_oracle(fgq, cuda_dev, M, N, K):
    a = fgq_inputs.exponent_spread((M, K), 20, 1, seed=M + 3)
    b = fgq_inputs.exponent_spread((K, N), 20, 128, seed=M + 4)
    host = _quant(a, b)
    ta, tb = _host_tiles(host)
    ga = fgq.ue8m0_scale_tiles(torch.from_numpy(host[1]).to(cuda_dev), weight=False)
    gb = fgq.ue8m0_scale_tiles(torch.from_numpy(host[3]).to(cuda_dev), weight=True)
    torch.cuda.synchronize()
    ma, mb = _defined(M, K), _defined(N, K)
    assert np.array_equal(ga.cpu().numpy()[ma], ta[ma])
    assert np.array_equal(gb.cpu().numpy()[mb], tb[mb])


# one row tile (single CTAs), pairs on 128- and 256-column tiles, a ragged
# and an odd number of row tiles, K/128 not a multiple of 4 (padded code
# cells), one chunk
TILED_SHAPES = [(33, 384, 640), (128, 256, 128), (300, 640, 1152), (1000, 512, 1024),
                (1100, 5120, 1536), (1280, 4096, 640), (2560, 2048, 2304)]


@pytest.mark.parametrize("M,N,K", TILED_SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_ue8m0_tiled_gemm(fgq, cuda_dev, M, N, K, out_dtype):
    """The code-tile GEMM against the oracle (sampled outputs plus the first
    and last 256 x 256 blocks whole), and bit for bit against the UE8M0
    path of fgq_gemm_fp8_blockscaled_ex on the same operands."""
    a = fgq_inputs.exponent_spread((M, K), 12, 1, seed=M + K)
    b = fgq_inputs.exponent_spread((K, N), 12, 128, seed=M + K + 1)
    host = _quant(a, b)
    ta, tb = _host_tiles(host)
    ops = _dev(*host, cuda_dev)
    c = fgq.gemm_fp8_ue8m0_tiled(ops[0], torch.from_numpy(ta).to(cuda_dev), ops[2],
                                 torch.from_numpy(tb).to(cuda_dev), out_dtype=out_dtype)
    c_ex = fgq.gemm_fp8_blockscaled(*ops, out_dtype=out_dtype, mode="ue8m0")
    torch.cuda.synchronize()
    m_last = ((M - 1) // 256) * 256
    blocks = [(r, q) for r0, q0 in ((0, 0), (m_last, max(N - 256, 0)))
              for r in range(r0, min(r0 + 256, M)) for q in range(q0, min(q0 + 256, N))]
    rng = np.random.default_rng(K)
    rows = np.concatenate([np.array([x[0] for x in blocks]), rng.integers(0, M, 2000)])
    cols = np.concatenate([np.array([x[1] for x in blocks]), rng.integers(0, N, 2000)])
    _check(c, host, rows, cols)
    assert torch.equal(c, c_ex)
    assert fgq.device_error() == 0


def test_ue8m0_tiled_large_prefill_from_the_gpu(fgq, cuda_dev):
    """4096 x 7168 x 7168, bf16 out, as the benchmark runs it: both operands
    quantized in one launch (UE8M0), code tiles made on the GPU, then the
    tiled GEMM; bit for bit the _ex UE8M0 result, and sampled outputs
    against the oracle."""
    M, N, K = 4096, 7168, 7168
    a, w = fgq_inputs.large_prefill(seed=0)
    xq, sx, wq, sw = fgq.quant_operands(a.to(cuda_dev), w.to(cuda_dev), "ue8m0")
    ta = fgq.ue8m0_scale_tiles(sx, weight=False)
    tb = fgq.ue8m0_scale_tiles(sw, weight=True)
    c = fgq.gemm_fp8_ue8m0_tiled(xq, ta, wq, tb, out_dtype=torch.bfloat16)
    c_ex = fgq.gemm_fp8_blockscaled(xq, sx, wq, sw, out_dtype=torch.bfloat16, mode="ue8m0")
    torch.cuda.synchronize()
    assert torch.equal(c, c_ex)
    host = (xq.cpu().numpy(), sx.cpu().numpy(), np.ascontiguousarray(wq.cpu().numpy().T),
            sw.cpu().numpy())
    rng = np.random.default_rng(2)
    rows = np.concatenate([rng.integers(0, M, 3000), [0, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 3000), [N - 1, 0]])
    _check(c, host, rows, cols)
    assert fgq.device_error() == 0


@pytest.mark.parametrize("M,N,K", [(300, 1024, 1536), (33, 384, 640), (4096, 7168, 7168)])
def test_quant_operands_ue8m0_tiles(fgq, cuda_dev, M, N, K):
    """The one-launch quantizer writing code tiles: codes as quant_operands
    in UE8M0 mode, scale codes bit for bit the oracle's in the tiled layout;
    and the tiled GEMM on them gives _ex's bits."""
    a, w = fgq_inputs.large_prefill(seed=5, m=M, k=K, n=N)
    xq, ta, wq, tb = fgq.quant_operands_ue8m0_tiles(a.to(cuda_dev), w.to(cuda_dev))
    xq2, sx, wq2, sw = fgq.quant_operands(a.to(cuda_dev), w.to(cuda_dev), "ue8m0")
    torch.cuda.synchronize()
    assert torch.equal(xq, xq2) and torch.equal(wq, wq2)
    host = (xq2.cpu().numpy(), sx.cpu().numpy(), np.ascontiguousarray(wq2.cpu().numpy().T),
            sw.cpu().numpy())
    oa, ow = oracle.quant_act_1x128(a, UE8M0), oracle.quant_w_128x128(w, UE8M0)
    assert np.array_equal(host[1], oa[1]) and np.array_equal(host[3], ow[1])
    ea, eb = _host_tiles(host)
    ma, mb = _defined(M, K), _defined(N, K)
    assert np.array_equal(ta.cpu().numpy()[ma], ea[ma])
    assert np.array_equal(tb.cpu().numpy()[mb], eb[mb])
    c = fgq.gemm_fp8_ue8m0_tiled(xq, ta, wq, tb, out_dtype=torch.bfloat16)
    c_ex = fgq.gemm_fp8_blockscaled(xq2, sx, wq2, sw, out_dtype=torch.bfloat16, mode="ue8m0")
    torch.cuda.synchronize()
    assert torch.equal(c, c_ex)
    assert fgq.device_error() == 0


@pytest.mark.parametrize("M,N,K", [(120, 384, 512), (600, 2560, 1024)], ids=["single", "pair"])
def test_ue8m0_tiled_padded_c(fgq, cuda_dev, M, N, K):
    """C as rows of a wider buffer (ldc > N, NaN canaries past column N)."""
    a = fgq_inputs.exponent_spread((M, K), 8, 1, seed=M)
    b = fgq_inputs.exponent_spread((K, N), 8, 128, seed=M + 9)
    host = _quant(a, b)
    ta, tb = _host_tiles(host)
    ops = _dev(*host, cuda_dev)
    buf = torch.full((M, N + 64), float("nan"), dtype=torch.bfloat16, device=cuda_dev)
    c = fgq.gemm_fp8_ue8m0_tiled(ops[0], torch.from_numpy(ta).to(cuda_dev), ops[2],
                                 torch.from_numpy(tb).to(cuda_dev), out_dtype=torch.bfloat16,
                                 out=buf[:, :N])
    torch.cuda.synchronize()
    assert torch.isnan(buf[:, N:].float()).all(), "the GEMM wrote past column N"
    _check(c, host)
