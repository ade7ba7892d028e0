"""The failure path of the kernels' bounded waits, on the GPU, without a
fault: a wait on a barrier that nothing completes gives up after its limit,
the device error word reports it through the C ABI, and the context stays
usable for the next call."""
import time

import numpy as np
import pytest
import torch

import fgq_inputs
import oracle

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_is_reported(fgq, cuda_dev):
    from fine_grained_fp8_gb300 import _lib
    assert fgq.device_error() == 0
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.monotonic()
    assert _lib.fgq_selftest_wait_timeout(stream) == _lib.FGQ_OK
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    st, word = _lib.fgq_device_error(True)
    assert st == _lib.FGQ_ERR_DEVICE_TIMEOUT
    assert word & 0x80, f"self-test bit not set: {word:#x}"
    assert 1.0 < waited < 60.0, f"the wait gave up after {waited:.2f} s"
    # cleared by the read above
    st, word = _lib.fgq_device_error(True)
    assert st == _lib.FGQ_OK and word == 0

    # the context still works: a small GEMM afterwards is within the bound
    a, b = fgq_inputs.tiny(seed=0)
    aq, sa = oracle.quant_act_1x128(a)
    bq, sb = oracle.quant_w_128x128(b)
    ops = (torch.from_numpy(aq).to(cuda_dev), torch.from_numpy(sa).to(cuda_dev),
           torch.from_numpy(np.ascontiguousarray(bq.T)).to(cuda_dev),
           torch.from_numpy(sb).to(cuda_dev))
    c = fgq.gemm_fp8_blockscaled(*ops)
    torch.cuda.synchronize()
    cref, tref = oracle.gemm_dequant(aq, sa, bq, sb)
    ok, ratio = oracle.gemm_within_tolerance(c.cpu().numpy().astype(np.float64), cref, tref, 2e-3)
    assert ok, f"max |err|/T = {ratio:.3e}"
    assert fgq.device_error() == 0
