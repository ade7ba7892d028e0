"""Parity of the sm_103a block-scaled FP8 GEMM with the oracle.

The bar ("Fine-Grained FP8/FP4 Quantization", §DeepGEMM): every fp32
accumulator satisfies
    |C - C_ref| <= 2e-3 * sum_k |a_hat[m,k]| |b_hat[k,n]|
where C_ref is the fp64 product of the dequantised operands; a bf16 output
may differ from that accumulator by its own rounding, half a bf16 ulp
(2^-8 of the value), which the bf16 cases add to the bound.  Every case is
compared element by element against the oracle on the whole output; the
full-size ones spread the oracle over the host's cores (oracle.threads).
The workloads' own configurations (tiny, outlier, large prefill, skinny)
run the whole path: the GPU quantizers on the workload's inputs, checked
bit for bit against the oracle's codes and scales, then the GPU GEMM on
those codes.
"""
import numpy as np
import pytest
import torch

import fgq_inputs
import oracle
from oracle.threads import gemm_dequant_parallel

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _oracle_operands(a_cpu, b_cpu, mode):
    aq, sa = oracle.quant_act_1x128(a_cpu, mode)
    bq, sb = oracle.quant_w_128x128(b_cpu, mode)
    return aq, sa, bq, sb


def _to_dev(aq, sa, bq, sb, dev):
    """Oracle operands in the library's layout (weight codes [N, K])."""
    return (torch.from_numpy(aq).to(dev), torch.from_numpy(sa).to(dev),
            torch.from_numpy(np.ascontiguousarray(bq.T)).to(dev), torch.from_numpy(sb).to(dev))


def _run(fgq, ops, out_dtype, mode_name, out=None):
    c = fgq.gemm_fp8_blockscaled(*ops, out_dtype=out_dtype, mode=mode_name, out=out)
    torch.cuda.synchronize()
    return c


def _check_full(c_gpu, aq, sa, bq, sb):
    cref, tref = gemm_dequant_parallel(aq, sa, bq, sb)
    c = c_gpu.float().cpu().numpy().astype(np.float64)
    ok, ratio = oracle.gemm_within_tolerance(c, cref, tref, TOL,
                                             out_bf16=c_gpu.dtype == torch.bfloat16)
    assert ok, f"max |err|/T = {ratio:.3e} exceeds {TOL}"
    return ratio


def _gpu_quantized(fgq, a, b, mode, dev):
    """The GPU quantizers on the workload's bf16 inputs, their codes and
    scales checked bit for bit against the oracle's; returns the device
    operands and the oracle's host operands (weight codes logical [K, N])."""
    name, mid = mode
    aq, sa = fgq.quant_act_1x128(a.to(dev), name)
    bq, sb = fgq.quant_w_128x128(b.to(dev), name)
    torch.cuda.synchronize()
    host = _oracle_operands(a, b, mid)
    got = (aq.cpu().numpy(), sa.cpu().numpy(), np.ascontiguousarray(bq.cpu().numpy().T),
           sb.cpu().numpy())
    for g, h, what in zip(got, host, ("A codes", "A scales", "B codes", "B scales")):
        assert np.array_equal(g.view(np.uint8), h.view(np.uint8)), f"GPU {what} differ from the oracle"
    return (aq, sa, bq, sb), host


MODES = [("fp32", oracle.MODE_FP32), ("ue8m0", oracle.MODE_UE8M0)]


def test_tiny_config(fgq, cuda_dev):
    """A [128, 256], B [256, 128], N(0, 1), fp32 scales, fp32 C."""
    a, b = fgq_inputs.tiny(seed=0)
    host = _oracle_operands(a, b, oracle.MODE_FP32)
    c = _run(fgq, _to_dev(*host, cuda_dev), torch.float32, "fp32")
    _check_full(c, *host)


def test_tiny_config_whole_path(fgq, cuda_dev):
    """The tiny workload through the GPU quantizers and the GEMM."""
    a, b = fgq_inputs.tiny(seed=0)
    ops, host = _gpu_quantized(fgq, a, b, MODES[0], cuda_dev)
    c = _run(fgq, ops, torch.float32, "fp32")
    _check_full(c, *host)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_outlier_config(fgq, cuda_dev, mode):
    """M = N = K = 1024, N(0, 1) with 0.1% of entries x100, fp32 C: the GPU
    quantizers on the workload's own inputs, then the GEMM."""
    a, b = fgq_inputs.outlier_gemm(1024, seed=0)
    ops, host = _gpu_quantized(fgq, a, b, mode, cuda_dev)
    c = _run(fgq, ops, torch.float32, mode[0])
    _check_full(c, *host)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (17, 384, 256), (200, 128, 384),
                                   (300, 640, 128), (129, 256, 1024)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_ragged_small(fgq, cuda_dev, M, N, K, out_dtype):
    a = fgq_inputs.outlier((M, K), 1e-2, 100.0, seed=M)
    b = fgq_inputs.normal((K, N), 0.02, seed=N)
    host = _oracle_operands(a, b, oracle.MODE_FP32)
    c = _run(fgq, _to_dev(*host, cuda_dev), out_dtype, "fp32")
    _check_full(c, *host)


@pytest.mark.parametrize("M", [2432, 2400])
def test_wide_tile_path(fgq, cuda_dev, M):
    """Enough tiles (>= one per SM) for the 128 x 256 tile configuration,
    with a ragged last M tile; bf16 output into a padded C."""
    N, K = 2048, 256
    a = fgq_inputs.normal((M, K), 1.0, seed=1)
    b = fgq_inputs.normal((K, N), 0.02, seed=2)
    host = _oracle_operands(a, b, oracle.MODE_FP32)
    out = torch.full((M, N + 64), float("nan"), dtype=torch.bfloat16, device=cuda_dev)[:, :N]
    c = _run(fgq, _to_dev(*host, cuda_dev), torch.bfloat16, "fp32", out=out)
    _check_full(c, *host)
    pad = out.as_strided((M, 64), (N + 64, 1), storage_offset=N)
    assert torch.isnan(pad.float()).all(), "GEMM wrote outside C's rows"


@pytest.mark.parametrize("M,N,K,out_dtype", [(600, 10240, 384, torch.float32),
                                             (2431, 128 * 77, 512, torch.bfloat16),
                                             (257, 128 * 160, 256, torch.bfloat16)])
def test_pair_tile_path(fgq, cuda_dev, M, N, K, out_dtype):
    """Enough 256 x 128 tiles for the CTA-pair kernel (tcgen05 cta_group::2):
    ragged M (an odd number of 128-row tiles leaves the last pair's second
    CTA with rows past M only), N not a multiple of 256, padded C."""
    a = fgq_inputs.outlier((M, K), 1e-3, 100.0, seed=M)
    b = fgq_inputs.normal((K, N), 0.02, seed=N % 997)
    host = _oracle_operands(a, b, oracle.MODE_FP32)
    out = torch.full((M, N + 64), float("nan"), dtype=out_dtype, device=cuda_dev)[:, :N]
    c = _run(fgq, _to_dev(*host, cuda_dev), out_dtype, "fp32", out=out)
    _check_full(c, *host)
    pad = out.as_strided((M, 64), (N + 64, 1), storage_offset=N)
    assert torch.isnan(pad.float()).all(), "GEMM wrote outside C's rows"


@pytest.mark.parametrize("out_dtype,pad", [(torch.bfloat16, 8), (torch.float32, 4)],
                         ids=["bf16", "f32"])
@pytest.mark.parametrize("M,N", [(1000, 4096), (2432, 2048)], ids=["tile128", "tile256"])
def test_c_rows_16_byte_aligned_only(fgq, cuda_dev, out_dtype, pad, M, N):
    """C whose start and row pitch are 16-byte but not 32-byte aligned (the
    ABI's minimum): the kernel falls back from 32-byte to 16-byte stores."""
    K = 256
    a = fgq_inputs.normal((M, K), 1.0, seed=31)
    b = fgq_inputs.normal((K, N), 0.02, seed=32)
    host = _oracle_operands(a, b, oracle.MODE_FP32)
    ldc = N + pad
    esz = 2 if out_dtype == torch.bfloat16 else 4
    buf = torch.full((M * ldc + 64,), float("nan"), dtype=out_dtype, device=cuda_dev)
    off = 16 // esz  # start 16 bytes past a 512-byte boundary
    out = buf.as_strided((M, N), (ldc, 1), storage_offset=off)
    assert (out.data_ptr() % 32) == 16 and (ldc * esz) % 32 == 16
    c = _run(fgq, _to_dev(*host, cuda_dev), out_dtype, "fp32", out=out)
    _check_full(c, *host)
    pad_view = buf.as_strided((M, pad), (ldc, 1), storage_offset=off + N)
    assert torch.isnan(pad_view.float()).all(), "GEMM wrote outside C's rows"


def test_plain_c_abi_signature(fgq, cuda_dev):
    """fgq_gemm_fp8_blockscaled(A, sA, B, sB, C, M, N, K, stream): fp32 out."""
    from fine_grained_fp8_gb300 import _lib
    a, b = fgq_inputs.tiny(seed=3)
    host = _oracle_operands(a, b, oracle.MODE_FP32)
    aq, sa, bq, sb = _to_dev(*host, cuda_dev)
    c = torch.empty((128, 128), dtype=torch.float32, device=cuda_dev)
    st = _lib.fgq_gemm_fp8_blockscaled(aq.data_ptr(), sa.data_ptr(), bq.data_ptr(), sb.data_ptr(),
                                       c.data_ptr(), 128, 128, 256,
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    _check_full(c, *host)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_end_to_end_quantize_then_gemm(fgq, cuda_dev, mode):
    """GPU quantizers feeding the GPU GEMM (the whole hot path)."""
    a, b = fgq_inputs.outlier_gemm(512, seed=4)
    aq, sa = fgq.quant_act_1x128(a.to(cuda_dev), mode[0])
    bq, sb = fgq.quant_w_128x128(b.to(cuda_dev), mode[0])
    c = _run(fgq, (aq, sa, bq, sb), torch.float32, mode[0])
    host = _oracle_operands(a, b, mode[1])
    _check_full(c, *host)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_large_prefill_full_size(fgq, cuda_dev, mode):
    """A [4096, 7168] N(0,1), B [7168, 7168] N(0,0.02^2), bf16 C, through the
    GPU quantizers, in the configuration the benchmark times; every one of
    the 29.4 M outputs against the oracle."""
    a, b = fgq_inputs.large_prefill(seed=0)
    ops, host = _gpu_quantized(fgq, a, b, mode, cuda_dev)
    c = _run(fgq, ops, torch.bfloat16, mode[0])
    _check_full(c, *host)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
@pytest.mark.parametrize("M", [16, 64, 256])
def test_skinny_full_size(fgq, cuda_dev, mode, M):
    """M x N=24576 x K=1536, bf16 C (the low-M paths): the GPU quantizers on
    the workload's own inputs, then the GEMM, every output against the
    oracle."""
    a, b = fgq_inputs.skinny(M, seed=0)
    ops, host = _gpu_quantized(fgq, a, b, mode, cuda_dev)
    c = _run(fgq, ops, torch.bfloat16, mode[0])
    _check_full(c, *host)


def test_repeat_calls_are_deterministic(fgq, cuda_dev):
    a, b = fgq_inputs.outlier_gemm(1024, seed=5)
    ops = _to_dev(*_oracle_operands(a, b, oracle.MODE_FP32), cuda_dev)
    c1 = _run(fgq, ops, torch.float32, "fp32").clone()
    c2 = _run(fgq, ops, torch.float32, "fp32")
    assert torch.equal(c1, c2)


def test_no_device_error_after_gemms(fgq, cuda_dev):
    assert fgq.device_error() == 0
