"""Parity of the low-M GEMM path (M <= 256: swapped operands, whole tiles or
stream-K over a caller-owned workspace) with the oracle, under the same
bound as the other GEMM tests ("Fine-Grained FP8/FP4 Quantization",
§DeepGEMM): |C - C_ref| <= 2e-3 * sum_k |a_hat||b_hat| for the fp32
accumulator, plus half a bf16 ulp for bf16 outputs."""
import numpy as np
import pytest
import torch

import fgq_inputs
import oracle
from oracle.threads import gemm_dequant_parallel

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _operands(M, N, K, seed, mode=oracle.MODE_FP32):
    a = fgq_inputs.outlier((M, K), 1e-2, 100.0, seed)
    b = fgq_inputs.normal((K, N), 0.02, seed + 1)
    aq, sa = oracle.quant_act_1x128(a, mode)
    bq, sb = oracle.quant_w_128x128(b, mode)
    return aq, sa, bq, sb


def _dev(aq, sa, bq, sb, dev):
    return (torch.from_numpy(aq).to(dev), torch.from_numpy(sa).to(dev),
            torch.from_numpy(np.ascontiguousarray(bq.T)).to(dev), torch.from_numpy(sb).to(dev))


def _check(c_gpu, host, rows=None, cols=None):
    if rows is None:
        cref, tref = gemm_dequant_parallel(*host)
        c = c_gpu.float().cpu().numpy().astype(np.float64)
    else:
        cref, tref = oracle.gemm_dequant_at(*host, rows, cols)
        c = c_gpu.float().cpu().numpy()[rows, cols].astype(np.float64)
    ok, ratio = oracle.gemm_within_tolerance(c, cref, tref, TOL,
                                             out_bf16=c_gpu.dtype == torch.bfloat16)
    assert ok, f"max |err|/T = {ratio:.3e} exceeds {TOL}"


# M covers every padded width (16, 32, 64, 128, 256); K covers one batch of
# chunk partials, several, and a short last batch
SHAPES = [(1, 384, 512), (7, 128, 256), (16, 640, 384), (24, 384, 1536), (32, 256, 2304),
          (33, 256, 1024), (64, 384, 512), (100, 256, 384), (128, 512, 256), (200, 384, 640),
          (256, 256, 512)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_lowm_no_split(fgq, cuda_dev, M, N, K, out_dtype):
    host = _operands(M, N, K, seed=M)
    c = fgq.gemm_fp8_blockscaled(*_dev(*host, cuda_dev), out_dtype=out_dtype)
    torch.cuda.synchronize()
    _check(c, host)


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_lowm_splitk(fgq, cuda_dev, M, N, K, out_dtype):
    host = _operands(M, N, K, seed=M + 1)
    ops = _dev(*host, cuda_dev)
    ws = fgq.splitk_workspace(M, N, K)
    c1 = fgq.gemm_fp8_blockscaled_splitk(*ops, ws, out_dtype=out_dtype)
    c2 = fgq.gemm_fp8_blockscaled_splitk(*ops, ws, out_dtype=out_dtype)
    c3 = fgq.gemm_fp8_blockscaled_splitk(*ops, ws, out_dtype=out_dtype)
    torch.cuda.synchronize()
    _check(c1, host)
    # each call leaves the counters and flags at zero for the next: three
    # calls on one workspace agree bit for bit
    assert torch.equal(c1, c2) and torch.equal(c1, c3), \
        "stream-K result changed between calls on the same workspace"


@pytest.mark.parametrize("mode", [("fp32", oracle.MODE_FP32), ("ue8m0", oracle.MODE_UE8M0)],
                         ids=lambda m: m[0])
def test_lowm_long_k_crosses_scale_windows(fgq, cuda_dev, mode):
    """K = 40 chunks: the activation scales are staged in 16-chunk windows."""
    M, N, K = 48, 256, 40 * 128
    host = _operands(M, N, K, seed=5, mode=mode[1])
    ops = _dev(*host, cuda_dev)
    c = fgq.gemm_fp8_blockscaled(*ops, out_dtype=torch.float32, mode=mode[0])
    ws = fgq.splitk_workspace(M, N, K)
    cs = fgq.gemm_fp8_blockscaled_splitk(*ops, ws, out_dtype=torch.float32, mode=mode[0])
    torch.cuda.synchronize()
    _check(c, host)
    _check(cs, host)


def test_splitk_rejects_small_workspace(fgq, cuda_dev):
    from fine_grained_fp8_gb300 import _lib
    M, N, K = 16, 1024, 1024
    host = _operands(M, N, K, seed=9)
    aq, sa, bq, sb = _dev(*host, cuda_dev)
    st, need = _lib.fgq_gemm_splitk_workspace_size(M, N, K)
    assert st == 0 and need > 256
    ws = torch.zeros(need, dtype=torch.uint8, device=cuda_dev)
    c = torch.empty((M, N), dtype=torch.float32, device=cuda_dev)
    stream = torch.cuda.current_stream().cuda_stream
    assert _lib.fgq_gemm_fp8_blockscaled_splitk(aq.data_ptr(), sa.data_ptr(), bq.data_ptr(),
                                                sb.data_ptr(), c.data_ptr(), N, M, N, K, 0, 0,
                                                ws.data_ptr(), need - 1, stream) == 1
    assert _lib.fgq_gemm_fp8_blockscaled_splitk(aq.data_ptr(), sa.data_ptr(), bq.data_ptr(),
                                                sb.data_ptr(), c.data_ptr(), N, M, N, K, 0, 0,
                                                ws.data_ptr(), need, stream) == 0
    torch.cuda.synchronize()
    _check(c, host)


def test_lowm_repeated_calls_complete(fgq, cuda_dev):
    """Many back-to-back calls at the skinny size for every padded width:
    each finishes without a kernel giving up on a wait, and repeats agree."""
    N, K = 24576, 1536
    for M in (16, 32, 64):
        a, b = fgq_inputs.skinny(M, seed=3)
        aq, sa = fgq.quant_act_1x128(a.to(cuda_dev))
        bq, sb = fgq.quant_w_128x128(b.to(cuda_dev))
        ws = fgq.splitk_workspace(M, N, K)
        first = fgq.gemm_fp8_blockscaled(aq, sa, bq, sb, out_dtype=torch.bfloat16)
        for _ in range(30):
            c = fgq.gemm_fp8_blockscaled(aq, sa, bq, sb, out_dtype=torch.bfloat16)
            cs = fgq.gemm_fp8_blockscaled_splitk(aq, sa, bq, sb, ws, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert fgq.device_error() == 0, f"M={M}: a kernel gave up on a wait"
        assert torch.equal(c, first)
        assert torch.isfinite(cs.float()).all()


@pytest.mark.parametrize("M", [16, 32, 64, 256])
def test_skinny_full_size_splitk(fgq, cuda_dev, M):
    """M x N=24576 x K=1536, bf16 C: the stream-K path on the GPU-quantized
    skinny operands (192 column tiles: one whole wave, the rest shared out
    by K chunks), every output against the oracle."""
    a, b = fgq_inputs.skinny(M, seed=0)
    aq, sa = fgq.quant_act_1x128(a.to(cuda_dev))
    bq, sb = fgq.quant_w_128x128(b.to(cuda_dev))
    ws = fgq.splitk_workspace(M, 24576, 1536)
    c = fgq.gemm_fp8_blockscaled_splitk(aq, sa, bq, sb, ws, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    host = (aq.cpu().numpy(), sa.cpu().numpy(), np.ascontiguousarray(bq.cpu().numpy().T),
            sb.cpu().numpy())
    _check(c, host)


# Stream-K shapes for a GB300's 152 SMs (the schedule adapts to any count):
#   one tile past a whole wave; fewer tiles than SMs with long K (ten
#   ranges per tile, ranges crossing the 16-chunk scale windows); wide
#   accumulators (M in (64, 256]) split among fewer CTAs; a few tiles past a
#   wave with a short K.
SK_SHAPES = [(16, 128 * 153, 1536), (16, 128 * 8, 40 * 128), (48, 128 * 160, 1536),
             (100, 128 * 20, 2048), (200, 128 * 5, 3072), (256, 128 * 155, 1024),
             (7, 128 * 3, 64 * 128)]


@pytest.mark.parametrize("M,N,K", SK_SHAPES)
@pytest.mark.parametrize("mode", [("fp32", oracle.MODE_FP32), ("ue8m0", oracle.MODE_UE8M0)],
                         ids=lambda m: m[0])
def test_stream_k_shapes(fgq, cuda_dev, M, N, K, mode):
    host = _operands(M, N, K, seed=N % 1000 + M, mode=mode[1])
    ops = _dev(*host, cuda_dev)
    ws = fgq.splitk_workspace(M, N, K)
    out_dtype = torch.bfloat16 if M % 2 == 0 else torch.float32
    c1 = fgq.gemm_fp8_blockscaled_splitk(*ops, ws, out_dtype=out_dtype, mode=mode[0])
    c2 = fgq.gemm_fp8_blockscaled_splitk(*ops, ws, out_dtype=out_dtype, mode=mode[0])
    torch.cuda.synchronize()
    _check(c1, host)
    assert torch.equal(c1, c2)
    assert fgq.device_error() == 0


# The default entry point's cluster-pair split (no workspace): the tiles
# after the last whole wave, or all tiles when there are at most one per
# cluster, are split in K within clusters of two (odd chunk counts split
# unevenly); other shapes run whole tiles.  For a GB300's 152 SMs.
PAIR_SHAPES = [(16, 128 * 192, 1536), (32, 128 * 155, 640), (9, 128 * 3, 3 * 128),
               (16, 128 * 76, 256), (16, 128 * 252, 256), (16, 1024, 128), (30, 128 * 40, 8 * 128)]


@pytest.mark.parametrize("M,N,K", PAIR_SHAPES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_lowm_cluster_pair_split(fgq, cuda_dev, M, N, K, out_dtype):
    host = _operands(M, N, K, seed=N % 991 + M)
    ops = _dev(*host, cuda_dev)
    c1 = fgq.gemm_fp8_blockscaled(*ops, out_dtype=out_dtype)
    c2 = fgq.gemm_fp8_blockscaled(*ops, out_dtype=out_dtype)
    torch.cuda.synchronize()
    _check(c1, host)
    assert torch.equal(c1, c2), "the split result changed between calls"
    assert fgq.device_error() == 0


def test_no_device_error_after_lowm(fgq, cuda_dev):
    assert fgq.device_error() == 0
