"""The GEMM that quantizes its bf16 activations itself (fused quantize ->
GEMM, few rows of A).

Its codes and scales are those of fgq_quant_act_1x128 and its GEMM is the
low-M kernel, so the result must equal, bit for bit, the quantizer followed
by fgq_gemm_fp8_blockscaled_ex (which takes the same kernel for M <= 32);
it is also held to the GEMM bound against the oracle ("Fine-Grained
FP8/FP4 Quantization", §DeepGEMM)."""
import numpy as np
import pytest
import torch

import fgq_inputs
import oracle

pytestmark = pytest.mark.gpu

MODES = [("fp32", oracle.MODE_FP32), ("ue8m0", oracle.MODE_UE8M0)]


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("M,N,K,pad", [(1, 384, 640, 0), (7, 128, 128, 8), (16, 1024, 1536, 0),
                                       (16, 256, 7936, 0), (17, 640, 1536, 64), (32, 384, 3968, 0)])
def test_fused_equals_quantizer_then_gemm(fgq, cuda_dev, mode, out_dtype, M, N, K, pad):
    a = fgq_inputs.outlier((M, K), 1e-2, 100.0, seed=M + K)
    if pad:
        big = torch.zeros((M, K + pad), dtype=torch.bfloat16)
        big[:, :K] = a
        a_dev = big.to(cuda_dev)[:, :K]
    else:
        a_dev = a.to(cuda_dev)
    b = fgq_inputs.normal((K, N), 0.02, seed=N)
    bq, sb = fgq.quant_w_128x128(b.to(cuda_dev), mode[0])
    c_fused = fgq.gemm_fp8_blockscaled_fused_act(a_dev, bq, sb, out_dtype=out_dtype, mode=mode[0])
    aq, sa = fgq.quant_act_1x128(a_dev.contiguous(), mode[0])
    c_ref = fgq.gemm_fp8_blockscaled(aq, sa, bq, sb, out_dtype=out_dtype, mode=mode[0])
    torch.cuda.synchronize()
    assert torch.equal(c_fused, c_ref), "fused result differs from quantizer + GEMM"
    if K <= 1536:
        # and within the bound against the oracle's fp64 product
        aqo, sao = oracle.quant_act_1x128(a, mode[1])
        bqo, sbo = oracle.quant_w_128x128(b, mode[1])
        cref, tref = oracle.gemm_dequant(aqo, sao, bqo, sbo)
        ok, ratio = oracle.gemm_within_tolerance(c_fused.float().cpu().numpy().astype(np.float64),
                                                 cref, tref, 2e-3,
                                                 out_bf16=out_dtype == torch.bfloat16)
        assert ok, f"max |err|/T = {ratio:.3e}"


def test_fused_skinny_full_size_repeated(fgq, cuda_dev):
    """M = 16 x N = 24576 x K = 1536, bf16 out, 20 calls in a row: all equal
    to the unfused path and no kernel gives up on a wait."""
    a, b = fgq_inputs.skinny(16, seed=4)
    a = a.to(cuda_dev)
    bq, sb = fgq.quant_w_128x128(b.to(cuda_dev))
    aq, sa = fgq.quant_act_1x128(a)
    ref = fgq.gemm_fp8_blockscaled(aq, sa, bq, sb, out_dtype=torch.bfloat16)
    for _ in range(20):
        c = fgq.gemm_fp8_blockscaled_fused_act(a, bq, sb, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(c, ref)
    assert fgq.device_error() == 0


@pytest.mark.parametrize("M,K", [(33, 1536), (16, 8064), (32, 4096)])
def test_fused_rejects_what_does_not_fit(fgq, cuda_dev, M, K):
    from fine_grained_fp8_gb300 import _lib
    N = 256
    a = torch.zeros((M, K), dtype=torch.bfloat16, device=cuda_dev)
    bq = torch.zeros((N, K), dtype=torch.uint8, device=cuda_dev)
    sb = torch.ones((K // 128, N // 128), dtype=torch.float32, device=cuda_dev)
    c = torch.empty((M, N), dtype=torch.float32, device=cuda_dev)
    rc = _lib.fgq_gemm_fp8_blockscaled_fused_act(a.data_ptr(), K, bq.data_ptr(), sb.data_ptr(),
                                                 c.data_ptr(), N, M, N, K, 0, 0,
                                                 torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.FGQ_ERR_INVALID_ARG
