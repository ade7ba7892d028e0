"""Parity of the sm_103a quantizers with the oracle: E4M3 codes and scales
must match bit for bit (the page's 1x128 / 128x128 granularities,
"Fine-Grained FP8/FP4 Quantization" §Scaling Granularities)."""
import numpy as np
import pytest
import torch

import fgq_inputs
import oracle
from golden_io import quant_groups

pytestmark = pytest.mark.gpu

MODES = [("fp32", oracle.MODE_FP32), ("ue8m0", oracle.MODE_UE8M0)]


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _assert_act_parity(fgq, x_cpu, mode, dev, ldx=None, ldq=None):
    name, mid = mode
    M, K = x_cpu.shape
    if ldx is None:
        x = x_cpu.to(dev)
    else:
        big = torch.zeros((M, ldx), dtype=torch.bfloat16, device=dev)
        big[:, :K] = x_cpu.to(dev)
        x = big[:, :K]
    xq = sx = None
    if ldq is not None:
        xq = torch.full((M, ldq), 0xA5, dtype=torch.uint8, device=dev)[:, :K]
    xq, sx = fgq.quant_act_1x128(x, name, xq=xq)
    torch.cuda.synchronize()
    oq, os_ = oracle.quant_act_1x128(x_cpu, mid)
    got_q = xq.cpu().numpy()
    got_s = sx.cpu().numpy()
    assert np.array_equal(got_s.view(np.uint32), os_.view(np.uint32)), "scales differ"
    if not np.array_equal(got_q, oq):
        bad = np.argwhere(got_q != oq)
        m, k = bad[0]
        raise AssertionError(
            f"{len(bad)} codes differ; first at ({m},{k}): x bits {_bits(x_cpu)[m, k]:#06x} "
            f"gpu {got_q[m, k]:#04x} oracle {oq[m, k]:#04x} scale {os_[m, k // 128]!r}")
    if ldq is not None:
        pad = xq.as_strided((M, ldq - K), (ldq, 1), storage_offset=K).cpu().numpy()
        assert np.all(pad == 0xA5), "quantizer wrote outside its rows"


def _assert_w_parity(fgq, w_cpu, mode, dev, ldw=None):
    name, mid = mode
    K, N = w_cpu.shape
    if ldw is None:
        w = w_cpu.to(dev)
    else:
        big = torch.zeros((K, ldw), dtype=torch.bfloat16, device=dev)
        big[:, :N] = w_cpu.to(dev)
        w = big[:, :N]
    wq, sw = fgq.quant_w_128x128(w, name)
    torch.cuda.synchronize()
    assert wq.shape == (N, K)
    oq, os_ = oracle.quant_w_128x128(w_cpu, mid)
    assert np.array_equal(sw.cpu().numpy().view(np.uint32), os_.view(np.uint32)), "scales differ"
    got = wq.cpu().numpy().T
    if not np.array_equal(got, oq):
        bad = np.argwhere(got != oq)
        raise AssertionError(f"{len(bad)} weight codes differ; first at {tuple(bad[0])}")


@pytest.mark.parametrize("case", quant_groups(), ids=lambda c: f"{c[0]}-{c[1]}")
def test_act_golden_groups(fgq, cuda_dev, case):
    """Hand-worked groups (tests/golden/quant_groups.txt) on the GPU."""
    name, mode, bits, scale_bits, codes = case
    x = np.zeros((2, 256), dtype=np.uint16)
    x[1, 128:128 + len(bits)] = bits  # group (1, 1); the others are all zero
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    xq, sx = fgq.quant_act_1x128(xt.to(cuda_dev), mode)
    torch.cuda.synchronize()
    s = sx.cpu().numpy().view(np.uint32)
    assert s[1, 1] == scale_bits
    assert np.all(s[0] == 0x3F800000) and s[1, 0] == 0x3F800000  # zero groups: scale 1
    want = np.zeros(128, dtype=np.uint8)
    want[:len(codes)] = codes
    q = xq.cpu().numpy()
    assert np.array_equal(q[1, 128:], want)
    assert np.all(q[0] == 0) and np.all(q[1, :128] == 0)


@pytest.mark.parametrize("case", quant_groups(), ids=lambda c: f"{c[0]}-{c[1]}")
def test_weight_golden_groups(fgq, cuda_dev, case):
    name, mode, bits, scale_bits, codes = case
    w = np.zeros((256, 128), dtype=np.uint16)
    pos = [(128 + (7 * i + 3) % 128, (5 * i + 11) % 128) for i in range(len(bits))]
    for (r, c), b in zip(pos, bits):
        w[r, c] = b
    wt = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16)
    wq, sw = fgq.quant_w_128x128(wt.to(cuda_dev), mode)
    torch.cuda.synchronize()
    s = sw.cpu().numpy().view(np.uint32)
    assert s[1, 0] == scale_bits and s[0, 0] == 0x3F800000
    q = wq.cpu().numpy()  # [N, K]
    for (r, c), code in zip(pos, codes):
        assert q[c, r] == code


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_act_every_bf16_pattern(fgq, cuda_dev, mode):
    """All 65536 bf16 bit patterns (NaN/Inf replaced by 0), 128 consecutive
    patterns per group: every magnitude, sign and subnormal, under scales
    from the smallest subnormal to the largest."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    nonfinite = (bits & 0x7F80) == 0x7F80
    bits[nonfinite] = 0
    x = torch.from_numpy(bits.view(np.int16).reshape(256, 256)).view(torch.bfloat16)
    _assert_act_parity(fgq, x, mode, cuda_dev)
    # the same values shuffled so each group mixes magnitudes
    perm = np.random.default_rng(3).permutation(65536)
    xs = torch.from_numpy(bits[perm].view(np.int16).reshape(512, 128)).view(torch.bfloat16)
    _assert_act_parity(fgq, xs, mode, cuda_dev)


def _every_x_below_amax(exponents):
    """Groups [amax, x1 .. x127]: for each bf16 amax with one of the given
    exponent fields and each of the 128 significands, every bf16 x with
    |x| <= amax, both signs, spread over as many groups as needed."""
    rows = []
    for e in exponents:
        for ma in range(128):
            amax = (e << 7) | ma
            mags = np.arange(0, amax + 1, dtype=np.uint32)
            xs = np.concatenate([mags, mags | 0x8000]).astype(np.uint16)
            pad = (-len(xs)) % 127
            xs = np.concatenate([xs, np.zeros(pad, np.uint16)]).reshape(-1, 127)
            head = np.full((xs.shape[0], 1), amax, np.uint16)
            rows.append(np.concatenate([head, xs], axis=1))
    bits = np.concatenate(rows)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
@pytest.mark.parametrize("exponent", [250, 127, 36, 35, 34, 1])
def test_act_every_x_for_every_amax_significand(fgq, cuda_dev, mode, exponent):
    """Within a group only amax's significand (128 values) and exponent fix
    the scale, so this covers every reachable (scale, x) pair of that amax
    binade: huge, ordinary, both sides of the 2^-100 scale boundary where
    the kernel switches to IEEE division, and the smallest normal binade."""
    x = _every_x_below_amax([exponent])
    _assert_act_parity(fgq, x, mode, cuda_dev)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
@pytest.mark.parametrize("M,K", [(1, 128), (3, 256), (129, 640), (1000, 1024), (77, 7168),
                                 (4096, 384)])
def test_act_shapes(fgq, cuda_dev, mode, M, K):
    x = fgq_inputs.student_t((M, K), 3, 1.0, seed=M + K)
    _assert_act_parity(fgq, x, mode, cuda_dev)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_act_outliers_and_strides(fgq, cuda_dev, mode):
    x = fgq_inputs.outlier((300, 1024), 1e-3, 100.0, seed=7)
    _assert_act_parity(fgq, x, mode, cuda_dev, ldx=1096, ldq=1040)
    _assert_act_parity(fgq, x, mode, cuda_dev, ldx=1024, ldq=1152)


def test_act_empty(fgq, cuda_dev):
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device=cuda_dev)
    xq, sx = fgq.quant_act_1x128(x)
    assert xq.shape == (0, 256) and sx.shape == (0, 2)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
@pytest.mark.parametrize("K,N,seed", [(128, 128, 1), (256, 384, 2), (1024, 1024, 3),
                                      (1536, 640, 4)])
def test_weight_shapes(fgq, cuda_dev, mode, K, N, seed):
    w = fgq_inputs.normal((K, N), 0.02, seed)
    _assert_w_parity(fgq, w, mode, cuda_dev)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_weight_outliers_and_stride(fgq, cuda_dev, mode):
    w = fgq_inputs.outlier((1024, 1024), 1e-3, 100.0, seed=9)
    _assert_w_parity(fgq, w, mode, cuda_dev, ldw=1160)
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    bits[(bits & 0x7F80) == 0x7F80] = 0
    wb = torch.from_numpy(bits.view(np.int16).reshape(256, 256)).view(torch.bfloat16)
    _assert_w_parity(fgq, wb, mode, cuda_dev)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_full_size_quant_bw_config(fgq, cuda_dev, mode):
    """The quantize-bandwidth workload at full size, every code and scale:
    activations [16384, 7168] Student-t (nu = 3), weight [7168, 7168]
    N(0, 0.02^2)."""
    a, w = fgq_inputs.quant_bw(seed=0)
    _assert_act_parity(fgq, a, mode, cuda_dev)
    _assert_w_parity(fgq, w, mode, cuda_dev)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_full_size_skinny_weight(fgq, cuda_dev, mode):
    _, w = fgq_inputs.skinny(16, seed=0)
    _assert_w_parity(fgq, w, mode, cuda_dev)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_tiny_config_quantizers(fgq, cuda_dev, mode):
    """The tiny workload's own inputs: A [128, 256] and B [256, 128], N(0, 1)."""
    a, b = fgq_inputs.tiny(seed=0)
    _assert_act_parity(fgq, a, mode, cuda_dev)
    _assert_w_parity(fgq, b, mode, cuda_dev)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_outlier_config_quantizers(fgq, cuda_dev, mode):
    """The outlier workload's own inputs, both scale modes: A and B [1024,
    1024] N(0, 1) with 0.1% of entries x100 at seeded positions."""
    a, b = fgq_inputs.outlier_gemm(1024, seed=0)
    _assert_act_parity(fgq, a, mode, cuda_dev)
    _assert_w_parity(fgq, b, mode, cuda_dev)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
@pytest.mark.parametrize("M", [16, 64, 256])
def test_skinny_config_activations(fgq, cuda_dev, mode, M):
    """The skinny sweep's own activations, A [M, 1536] N(0, 1) (its weight
    is covered by test_full_size_skinny_weight)."""
    a, _ = fgq_inputs.skinny(M, seed=0)
    _assert_act_parity(fgq, a, mode, cuda_dev)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
@pytest.mark.parametrize("M,K,N", [(0, 256, 384), (1, 128, 128), (129, 640, 256), (77, 7168, 1024),
                                   (4096, 7168, 7168)])
def test_quant_operands_one_launch(fgq, cuda_dev, mode, M, K, N):
    """Both operands in one launch: codes and scales bit for bit those of the
    oracle (and so of the two separate quantizers), including an empty A and
    the large-prefill operands."""
    name, mid = mode
    a = fgq_inputs.student_t((M, K), 3, 1.0, seed=M + 1) if M else torch.zeros((0, K), dtype=torch.bfloat16)
    w = fgq_inputs.normal((K, N), 0.02, seed=N + 2)
    xq, sx, wq, sw = fgq.quant_operands(a.to(cuda_dev), w.to(cuda_dev), name)
    torch.cuda.synchronize()
    if M:
        oq, os_ = oracle.quant_act_1x128(a, mid)
        assert np.array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))
        assert np.array_equal(xq.cpu().numpy(), oq)
    wo, wso = oracle.quant_w_128x128(w, mid)
    assert np.array_equal(sw.cpu().numpy().view(np.uint32), wso.view(np.uint32))
    assert np.array_equal(wq.cpu().numpy().T, wo)


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m[0])
def test_quant_operands_strided(fgq, cuda_dev, mode):
    """Strided activations and weight, padded code rows: the same bits as the
    separate quantizers, and nothing written outside the codes' rows."""
    name, _ = mode
    M, K, N = 300, 1024, 640
    a = fgq_inputs.outlier((M, K), 1e-3, 100.0, seed=11)
    w = fgq_inputs.outlier((K, N), 1e-3, 100.0, seed=12)
    abig = torch.zeros((M, K + 72), dtype=torch.bfloat16, device=cuda_dev)
    abig[:, :K] = a.to(cuda_dev)
    wbig = torch.zeros((K, N + 136), dtype=torch.bfloat16, device=cuda_dev)
    wbig[:, :N] = w.to(cuda_dev)
    xq = torch.full((M, K + 16), 0xA5, dtype=torch.uint8, device=cuda_dev)[:, :K]
    xq, sx, wq, sw = fgq.quant_operands(abig[:, :K], wbig[:, :N], name, xq=xq)
    xq2, sx2 = fgq.quant_act_1x128(abig[:, :K], name)
    wq2, sw2 = fgq.quant_w_128x128(wbig[:, :N], name)
    torch.cuda.synchronize()
    assert torch.equal(xq, xq2) and torch.equal(sx.view(torch.int32), sx2.view(torch.int32))
    assert torch.equal(wq, wq2) and torch.equal(sw.view(torch.int32), sw2.view(torch.int32))
    pad = xq.as_strided((M, 16), (K + 16, 1), storage_offset=K)
    assert bool((pad == 0xA5).all()), "quantizer wrote outside its rows"


def test_no_device_error(fgq, cuda_dev):
    assert fgq.device_error() == 0
