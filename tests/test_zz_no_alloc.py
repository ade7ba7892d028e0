"""The split-K GEMM entry point that allocates nothing.

Some callers cannot allocate device memory (code inside an allocator or a
memory-pool callback, hosts that give a library a fixed device-memory
budget up front), so fgq_gemm_fp8_blockscaled_splitk_noalloc keeps its
split-K scratch in a fixed array inside the library instead of a caller
workspace.  This file checks, through the C ABI, that two calls in a row
give the same output as the existing entry points, within the GEMM tests'
tolerance, that they leave the device's free memory unchanged, and that a
problem too large for the fixed array is refused.

It sits in a file of its own that pytest collects last, and passes both on
its own in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import fgq_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _operands(M, N, K, dev, seed=3, mode=oracle.MODE_FP32):
    a = fgq_inputs.outlier((M, K), 1e-2, 100.0, seed)
    b = fgq_inputs.normal((K, N), 0.02, seed + 1)
    aq, sa = oracle.quant_act_1x128(a, mode)
    bq, sb = oracle.quant_w_128x128(b, mode)
    host = (aq, sa, bq, sb)
    ops = (torch.from_numpy(aq).to(dev), torch.from_numpy(sa).to(dev),
           torch.from_numpy(np.ascontiguousarray(bq.T)).to(dev), torch.from_numpy(sb).to(dev))
    return host, ops


@pytest.mark.parametrize("M,N,K,out_dtype,mode,splits", [
    (16, 1024, 4096, torch.float32, oracle.MODE_FP32, True),
    (48, 1024, 3072, torch.bfloat16, oracle.MODE_FP32, True),
    (16, 24576, 512, torch.bfloat16, oracle.MODE_FP32, False),
    (200, 1024, 4096, torch.bfloat16, oracle.MODE_UE8M0, True),
], ids=["m16-f32-split", "m48-bf16-split", "m16-bf16-nosplit", "m200-bf16-ue8m0-split"])
def test_noalloc_matches_existing_entry_points(fgq, cuda_dev, M, N, K, out_dtype, mode, splits):
    from fine_grained_fp8_gb300 import _lib
    host, (aq, sa, bq, sb) = _operands(M, N, K, cuda_dev, mode=mode)
    st, need = _lib.fgq_gemm_splitk_workspace_size(M, N, K)
    assert st == 0
    # a case with partial tiles uses the scratch; one whose leftover tiles
    # divide evenly among the SMs has none and never touches it
    assert (need > 256) == splits
    assert need <= _lib.FGQ_NOALLOC_SCRATCH_BYTES
    out = _lib.FGQ_OUT_BF16 if out_dtype == torch.bfloat16 else _lib.FGQ_OUT_F32
    smode = _lib.FGQ_SCALE_UE8M0 if mode == oracle.MODE_UE8M0 else _lib.FGQ_SCALE_FP32
    stream = torch.cuda.current_stream().cuda_stream

    def call_noalloc(c):
        rc = _lib.fgq_gemm_fp8_blockscaled_splitk_noalloc(
            aq.data_ptr(), sa.data_ptr(), bq.data_ptr(), sb.data_ptr(), c.data_ptr(), N,
            M, N, K, out, smode, stream)
        assert rc == 0, _lib.status_string(rc)
        return c

    c0, c1, c2 = (torch.full((M, N), float("nan"), dtype=out_dtype, device=cuda_dev)
                  for _ in range(3))
    call_noalloc(c0)  # the first call on the device looks up the array's address
    torch.cuda.synchronize()
    # The promise is that a call allocates nothing: the device's free memory
    # and torch's allocator are unchanged across two more calls.
    free_before = torch.cuda.mem_get_info(cuda_dev)[0]
    torch_before = torch.cuda.memory_stats(cuda_dev)["allocation.all.allocated"]
    call_noalloc(c1)
    call_noalloc(c2)  # second call in a row: the shared scratch is reused
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(cuda_dev)[0] == free_before, "device memory was allocated"
    assert torch.cuda.memory_stats(cuda_dev)["allocation.all.allocated"] == torch_before
    c_ex = torch.empty((M, N), dtype=out_dtype, device=cuda_dev)
    assert _lib.fgq_gemm_fp8_blockscaled_ex(aq.data_ptr(), sa.data_ptr(), bq.data_ptr(),
                                            sb.data_ptr(), c_ex.data_ptr(), N, M, N, K, out,
                                            smode, stream) == 0
    ws = fgq.splitk_workspace(M, N, K)
    c_sk = torch.empty((M, N), dtype=out_dtype, device=cuda_dev)
    assert _lib.fgq_gemm_fp8_blockscaled_splitk(aq.data_ptr(), sa.data_ptr(), bq.data_ptr(),
                                                sb.data_ptr(), c_sk.data_ptr(), N, M, N, K, out,
                                                smode, ws.data_ptr(), ws.numel(),
                                                stream) == 0
    torch.cuda.synchronize()

    # against the existing entry point, within the tolerance of the GEMM
    # tests (each result is within it of the fp64 reference, so they are
    # within twice it of each other)
    cref, tref = oracle.gemm_dequant(*host)
    bf16 = out_dtype == torch.bfloat16
    for c in (c1, c2):
        ok, ratio = oracle.gemm_within_tolerance(c.float().cpu().numpy(), cref, tref, TOL,
                                                 out_bf16=bf16)
        assert ok, f"no-alloc output: max |err|/T = {ratio:.3e}"
    d = np.abs(c1.float().cpu().numpy() - c_ex.float().cpu().numpy())
    one = TOL * tref + (2.0 ** -8 * (np.abs(cref) + TOL * tref) if bf16 else 0.0)
    bound = 2 * one
    assert np.all(d <= bound), "no-alloc output differs from fgq_gemm_fp8_blockscaled_ex"
    # same kernel and schedule as the workspace entry point: identical bits,
    # and identical across the calls
    assert torch.equal(c0, c1) and torch.equal(c1, c2)
    assert torch.equal(c1, c_sk)
    assert fgq.device_error() == 0


def test_noalloc_refuses_problems_beyond_the_fixed_array(fgq, cuda_dev):
    from fine_grained_fp8_gb300 import _lib
    M, N, K = 256, 8192, 64 * 128
    st, need = _lib.fgq_gemm_splitk_workspace_size(M, N, K)
    assert st == 0
    if need <= 16 << 20:
        pytest.skip("this device splits the case little enough to fit the array")
    dummy = torch.zeros(16, dtype=torch.uint8, device=cuda_dev)
    p = dummy.data_ptr()
    rc = _lib.fgq_gemm_fp8_blockscaled_splitk_noalloc(p, p, p, p, p, N, M, N, K,
                                                      _lib.FGQ_OUT_F32, _lib.FGQ_SCALE_FP32,
                                                      torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.FGQ_ERR_INVALID_ARG
