"""Pins for the CPU oracle: facts that hold independently of its code.

Each test checks the oracle against something other than itself: values
the page prints or that follow by hand from the E4M3 / UE8M0 definitions
(tests/golden/), a library implementation of E4M3 (torch.float8_e4m3fn,
round-to-nearest-even on the finite range), closed forms, invariants, and
numpy's matmul on dequantised operands.  A plausible slip in the oracle (a
wrong rounding direction, a dropped sign, a transposed scale index, a
missing term) fails at least one of them.
"""
import math
import struct

import numpy as np
import pytest
import torch

import fgq_inputs
import oracle
from golden_io import e4m3_codes, quant_groups

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f32_bits(v):
    return struct.unpack("<I", struct.pack("<f", float(v)))[0]


def bits_f32(b):
    return struct.unpack("<f", struct.pack("<I", int(b)))[0]


# ---- E4M3 codec -----------------------------------------------------------

def test_e4m3_golden_codes():
    for code, value in e4m3_codes():
        got = oracle.e4m3_decode(code)
        if math.isnan(value):
            assert math.isnan(got), hex(code)
        else:
            assert got == value and math.copysign(1, got) == math.copysign(1, value), hex(code)
            assert oracle.e4m3_encode(value) == code, hex(code)


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_e4m3_roundtrip_and_monotone():
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    for c in finite:
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c
    pos = [oracle.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))
    assert max(pos) == 448.0


def _structured_fp32_values():
    """fp32 patterns around every rounding boundary of E4M3: every exponent
    from 2^-20 to 2^9, all top-11 mantissa bit patterns, and low bits at the
    tie point, just below and just above it, for both signs."""
    vals = []
    hi = np.arange(2048, dtype=np.uint32) << 12
    for lo in (0, 1, 0x7FF, 0x800, 0x801, 0xFFF):
        for e in range(127 - 20, 127 + 9):
            vals.append((np.uint32(e) << 23) | hi | np.uint32(lo))
    v = np.concatenate(vals)
    v = np.concatenate([v, v | np.uint32(0x80000000)])
    return v.view(np.float32)


def test_e4m3_encode_matches_torch_rne():
    x = _structured_fp32_values()
    x = x[np.abs(x) < 464.0]  # torch turns |x| >= 464 into NaN instead of saturating
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    enc = np.vectorize(oracle.e4m3_encode, otypes=[np.uint8])
    sample = np.random.default_rng(0).choice(x.size, size=min(x.size, 120000), replace=False)
    got = enc(x[sample])
    assert np.array_equal(got, ref[sample])


def test_e4m3_saturation_and_signed_zero():
    for v in (448.0, 449.0, 463.9, 464.0, 480.0, 1e30, 3.0e38):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-30) == 0x80
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00            # tie with 0 -> even
    assert oracle.e4m3_encode(2.0 ** -10 + 2.0 ** -30) == 0x01


def test_e4m3_midpoints_go_to_even_code():
    for c in range(0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = (lo + hi) / 2  # exact in fp32: E4M3 values have 4 significant bits
        assert float(np.float32(mid)) == mid
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == want
        assert oracle.e4m3_encode(-mid) == want | 0x80


# ---- scales -----------------------------------------------------------------

def _all_positive_finite_bf16():
    bits = np.arange(1, 0x7F80, dtype=np.uint32)  # +subnormals .. max finite
    return (bits << 16).view(np.float32)


def test_scale_fp32_puts_amax_on_448():
    """The group maximum always lands on E4M3 448 in fp32 mode: s is
    amax/448 rounded once, so amax/s is within an ulp of 448 (or above it
    and saturates), for every positive bf16 amax."""
    for amax in _all_positive_finite_bf16()[::7]:
        s = oracle.scale_from_amax(float(amax), oracle.MODE_FP32)
        assert s > 0 and math.isfinite(s)
        y = np.float32(amax) / np.float32(s)
        if s >= 2.0 ** -126:  # normal scale: one rounding, relative error <= 2^-24
            assert abs(float(y) - 448.0) <= 448.0 * 2.0 ** -22
        else:                 # subnormal scale (amax < ~2^-117): coarser, still nearest 448
            assert abs(float(y) - 448.0) < 16.0
        assert oracle.e4m3_encode(float(y)) == 0x7E


def test_scale_ue8m0_is_power_of_two_ceiling():
    for amax in _all_positive_finite_bf16()[::5]:
        t = float(np.float32(amax) / np.float32(448.0))
        s = oracle.scale_from_amax(float(amax), oracle.MODE_UE8M0)
        m, e = math.frexp(s)
        assert m == 0.5, s                       # power of two
        code = oracle.ue8m0_code(s)
        assert 0 <= code <= 254 and s == 2.0 ** (code - 127)
        if s > 2.0 ** -127:
            assert s >= t and s / 2 < t          # the smallest power >= t
        else:
            assert s >= t or s == 2.0 ** -127    # clamped at the bottom code


def test_scale_zero_group_and_closed_forms():
    for mode in (oracle.MODE_FP32, oracle.MODE_UE8M0):
        assert oracle.scale_from_amax(0.0, mode) == 1.0
    assert oracle.scale_from_amax(448.0, oracle.MODE_FP32) == 1.0
    assert oracle.scale_from_amax(224.0, oracle.MODE_FP32) == 0.5
    assert oracle.scale_from_amax(7.0, oracle.MODE_FP32) == 2.0 ** -6
    assert oracle.scale_from_amax(448.0, oracle.MODE_UE8M0) == 1.0
    assert oracle.scale_from_amax(450.0, oracle.MODE_UE8M0) == 2.0
    assert oracle.scale_from_amax(447.0, oracle.MODE_UE8M0) == 1.0
    assert oracle.pow2_ceil(1.0) == 1.0 and oracle.pow2_ceil(1.0000001) == 2.0
    assert oracle.pow2_ceil(0.75) == 1.0 and oracle.pow2_ceil(0.5) == 0.5


def test_ue8m0_pack_matches_page_formula():
    """Blackwell: Native Block Scaling: scale_i = 2^(((packed >> 8i) & 0xFF) - 127)."""
    codes = [127, 0, 254, 130]
    packed = oracle.ue8m0_pack4(codes)
    assert packed == 127 | (0 << 8) | (254 << 16) | (130 << 24)
    assert [oracle.ue8m0_unpack(packed, i) for i in range(4)] == [1.0, 2.0 ** -127, 2.0 ** 127, 8.0]
    assert oracle.ue8m0_code(1.0) == 127 and oracle.ue8m0_code(0.75) == -1


# ---- quantizers -----------------------------------------------------------

@pytest.mark.parametrize("case", quant_groups(), ids=lambda c: f"{c[0]}-{c[1]}")
def test_quant_act_golden_groups(case):
    name, mode, bits, scale_bits, codes = case
    mode_id = oracle.MODE_UE8M0 if mode == "ue8m0" else oracle.MODE_FP32
    x = np.zeros((1, 128), dtype=np.uint16)
    x[0, :len(bits)] = bits
    q, s = oracle.quant_act_1x128(x, mode_id)
    assert f32_bits(s[0, 0]) == scale_bits
    want = np.zeros(128, dtype=np.uint8)
    want[:len(codes)] = codes
    assert np.array_equal(q[0], want)


@pytest.mark.parametrize("case", quant_groups(), ids=lambda c: f"{c[0]}-{c[1]}")
def test_quant_w_golden_groups_as_blocks(case):
    """The same group laid out down a column of a 128x128 block (K direction)
    and scattered over rows gives the same scale and codes."""
    name, mode, bits, scale_bits, codes = case
    mode_id = oracle.MODE_UE8M0 if mode == "ue8m0" else oracle.MODE_FP32
    w = np.zeros((128, 128), dtype=np.uint16)
    pos = [(7 * i + 3) % 128 for i in range(len(bits))]
    for i, b in enumerate(bits):
        w[pos[i], (5 * i + 11) % 128] = b
    q, s = oracle.quant_w_128x128(w, mode_id)
    assert f32_bits(s[0, 0]) == scale_bits
    for i, c in enumerate(codes):
        assert q[pos[i], (5 * i + 11) % 128] == c
    mask = np.ones((128, 128), bool)
    for i in range(len(bits)):
        mask[pos[i], (5 * i + 11) % 128] = False
    assert np.all(q[mask] == 0)


def _ulp_e4m3(y):
    y = np.abs(y)
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    return np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))


@pytest.mark.parametrize("mode", [oracle.MODE_FP32, oracle.MODE_UE8M0])
def test_quant_act_invariants(mode):
    import fgq_inputs
    x = fgq_inputs.student_t((48, 640), 3, 1.0, seed=5)
    xo = fgq_inputs.outlier((16, 640), 1e-2, 100.0, seed=6)
    x = torch.cat([x, xo])
    x[3, 128:256] = 0
    xb = x.view(torch.int16).numpy().view(np.uint16)
    xf = x.float().numpy().astype(np.float64)
    q, s = oracle.quant_act_1x128(xb, mode)
    M, K = x.shape
    assert s.shape == (M, K // 128) and q.shape == (M, K)
    dec = oracle.e4m3_decode_array(q)
    assert np.all(np.isfinite(dec)) and np.all(np.abs(dec) <= 448)
    groups = xf.reshape(M, K // 128, 128)
    dq = dec.reshape(M, K // 128, 128)
    amax = np.abs(groups).max(axis=2)
    gmax = np.abs(dq).max(axis=2)
    nz = amax > 0
    if mode == oracle.MODE_FP32:
        assert np.all(gmax[nz] == 448)
        assert np.allclose(s[nz].astype(np.float64) * 448, amax[nz], rtol=2.0 ** -22, atol=0)
    else:
        assert np.all((gmax[nz] >= 224) & (gmax[nz] <= 448))
        m, _ = np.frexp(s)
        assert np.all(m == 0.5)
    assert np.all(s[~nz] == 1.0) and np.all(dq[~nz] == 0)
    # dequant error bound: half an E4M3 ulp of x/s, plus the fp32 rounding of x/s
    sc = np.repeat(s.astype(np.float64), 128, axis=1).reshape(M, K // 128, 128)
    y = groups / sc
    err = np.abs(y - dq)
    assert np.all(err <= 0.5 * _ulp_e4m3(y) + np.abs(y) * 2.0 ** -23)
    # sign: codes carry the sign of x, including for values that round to zero
    assert np.array_equal((q >= 0x80), np.signbit(xf.reshape(M, K)))


def test_quant_lossless_on_representable_groups():
    """A group made of E4M3 values times 2^j with a member at 448 * 2^j has
    scale 2^j in both modes and quantizes without loss."""
    rng = np.random.default_rng(1)
    pos = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    for j in (-8, 0, 5):
        vals = rng.choice(pos, size=(4, 256)) * rng.choice([-1.0, 1.0], size=(4, 256))
        vals[:, 0] = 448.0
        vals[:, 128] = -448.0
        x = torch.tensor(vals * 2.0 ** j, dtype=torch.float32)
        xb = x.to(torch.bfloat16)
        assert torch.equal(xb.float(), x)
        for mode in (oracle.MODE_FP32, oracle.MODE_UE8M0):
            q, s = oracle.quant_act_1x128(xb, mode)
            assert np.all(s == 2.0 ** j)
            assert np.array_equal(oracle.e4m3_decode_array(q) * 2.0 ** j, vals * 2.0 ** j)


def test_quant_w_block_indexing():
    """Each 128x128 block gets its own scale at sW[k/128, n/128]: blocks with
    distinct maxima (non-square block grid) land at the right index."""
    K, N = 256, 384
    w = np.zeros((K, N), dtype=np.float32)
    for i in range(K // 128):
        for j in range(N // 128):
            w[i * 128 + 17, j * 128 + 101] = 448.0 * 2.0 ** (i * 3 + j)
            w[i * 128 + 5, j * 128 + 9] = -1.0
    wb = torch.from_numpy(w).to(torch.bfloat16)
    q, s = oracle.quant_w_128x128(wb, oracle.MODE_FP32)
    assert s.shape == (2, 3)
    for i in range(2):
        for j in range(3):
            assert s[i, j] == 2.0 ** (i * 3 + j)
            assert q[i * 128 + 17, j * 128 + 101] == 0x7E


@pytest.mark.parametrize("mode", [oracle.MODE_FP32, oracle.MODE_UE8M0])
@pytest.mark.parametrize("kind", ["normal", "spread", "outlier"])
def test_quant_act_128x1_is_1x128_of_the_transpose(mode, kind):
    """Groups of 128 rows of one column of X are the 1x128 groups of X^T, so
    the transposed quantizer equals the (independently pinned) 1x128
    quantizer applied to X^T, in the same output layout, bit for bit."""
    import fgq_inputs
    M, K = 384, 256
    if kind == "normal":
        x = fgq_inputs.normal((M, K), 1.0, seed=1)
    elif kind == "spread":
        x = fgq_inputs.exponent_spread((M, K), 30, 128, seed=2)
    else:
        x = fgq_inputs.outlier((M, K), 1e-2, 100.0, seed=3)
    q, s = oracle.quant_act_128x1(x, mode)
    qt, st = oracle.quant_act_1x128(x.t().contiguous(), mode)
    assert q.shape == (K, M) and s.shape == (K, M // 128)
    assert np.array_equal(q, qt)
    assert np.array_equal(s.view(np.uint32), st.view(np.uint32))


def test_quant_act_128x1_group_indexing():
    """Group (k, mb) = rows 128 mb .. +127 of column k, its scale at sXT[k, mb]
    and the code of X[m, k] at XqT[k, m]: groups with distinct maxima on a
    non-square grid land where they belong."""
    M, K = 384, 256
    x = np.zeros((M, K), dtype=np.float32)
    for mb in range(M // 128):
        for k in (0, 5, 130, 255):
            x[mb * 128 + 77, k] = 448.0 * 2.0 ** (mb * 4 + k % 7)
            x[mb * 128 + 3, k] = -1.0
    xb = torch.from_numpy(x).to(torch.bfloat16)
    q, s = oracle.quant_act_128x1(xb, oracle.MODE_FP32)
    for mb in range(M // 128):
        for k in range(K):
            if k in (0, 5, 130, 255):
                assert s[k, mb] == 2.0 ** (mb * 4 + k % 7)
                assert q[k, mb * 128 + 77] == 0x7E
                assert q[k, mb * 128 + 3] != 0  # -1/s is a nonzero code for these scales
            else:
                assert s[k, mb] == 1.0      # all-zero group
                assert not q[k, mb * 128:(mb + 1) * 128].any()


def test_quant_rejects_bad_shapes_and_nonfinite():
    with pytest.raises(ValueError):
        oracle.quant_act_1x128(np.zeros((2, 100), np.uint16))
    with pytest.raises(ValueError):
        oracle.quant_w_128x128(np.zeros((128, 100), np.uint16))
    with pytest.raises(ValueError):
        oracle.quant_act_128x1(np.zeros((100, 128), np.uint16))
    x = np.zeros((1, 128), np.uint16)
    x[0, 3] = 0x7F80  # +inf
    with pytest.raises(ValueError):
        oracle.quant_act_1x128(x)


# ---- GEMM -------------------------------------------------------------------

def _dequant_with_torch(q, s, block_rows, block_cols):
    """Independent dequantisation: torch's E4M3 decode times the scale of
    each element's block, in fp64."""
    dec = torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()
    srep = np.repeat(np.repeat(s.astype(np.float64), block_rows, 0), block_cols, 1)
    return dec * srep


def _quantized_pair(M, N, K, seed, mode=oracle.MODE_FP32):
    import fgq_inputs
    a = fgq_inputs.outlier((M, K), 1e-2, 100.0, seed)
    b = fgq_inputs.normal((K, N), 0.02, seed + 1)
    aq, sa = oracle.quant_act_1x128(a, mode)
    bq, sb = oracle.quant_w_128x128(b, mode)
    return aq, sa, bq, sb


@pytest.mark.parametrize("mode", [oracle.MODE_FP32, oracle.MODE_UE8M0])
def test_gemm_matches_numpy_matmul_of_dequantised(mode):
    M, N, K = 40, 384, 256  # non-square block grid: kc = 2, nb = 3
    aq, sa, bq, sb = _quantized_pair(M, N, K, 11, mode)
    ah = _dequant_with_torch(aq, sa, 1, 128)
    bh = _dequant_with_torch(bq, sb, 128, 128)
    c, t = oracle.gemm_dequant(aq, sa, bq, sb)
    tref = np.abs(ah) @ np.abs(bh)
    assert np.all(np.abs(c - ah @ bh) <= 1e-12 * tref)
    assert np.allclose(t, tref, rtol=1e-12, atol=0)


def test_gemm_forms_agree_with_bruteforce():
    M, N, K = 8, 256, 384
    aq, sa, bq, sb = _quantized_pair(M, N, K, 21)
    c, t = oracle.gemm_dequant(aq, sa, bq, sb)
    cb = oracle.gemm_bruteforce(aq, sa, bq, sb)
    cc = oracle.gemm_chunked(aq, sa, bq, sb)
    scale = t + 1e-300
    assert np.all(np.abs(c - cb) <= 1e-13 * scale)
    assert np.all(np.abs(c - cc) <= 1e-13 * scale)
    rows = np.array([0, 7, 3, 5]); cols = np.array([0, 255, 128, 17])
    ca, ta = oracle.gemm_dequant_at(aq, sa, bq, sb, rows, cols)
    assert np.array_equal(ca, c[rows, cols]) and np.array_equal(ta, t[rows, cols])
    assert np.all(t >= np.abs(c))


def test_gemm_closed_forms():
    # constant operands: A = 448 (s = 1, code 0x7E), B = 7 (s = 2^-6, code 0x7E)
    M, N, K = 2, 128, 256
    a = torch.full((M, K), 448.0).to(torch.bfloat16)
    b = torch.full((K, N), 7.0).to(torch.bfloat16)
    aq, sa = oracle.quant_act_1x128(a)
    bq, sb = oracle.quant_w_128x128(b)
    c, t = oracle.gemm_dequant(aq, sa, bq, sb)
    assert np.all(c == K * 448.0 * 7.0) and np.all(t == c)
    # B = identity (128x128 blocks of I, all with scale 2^-7): C = A_hat / 2^... exactly
    K = N = 256
    a = fgq_inputs_normal((4, K), 3)
    bi = torch.eye(K, dtype=torch.float32).mul(448.0 * 2.0 ** -7).to(torch.bfloat16)
    aq, sa = oracle.quant_act_1x128(a)
    bq, sb = oracle.quant_w_128x128(bi)
    assert np.all(sb[np.eye(2, dtype=bool)] == 2.0 ** -7) and np.all(sb[~np.eye(2, dtype=bool)] == 1.0)
    c, _ = oracle.gemm_dequant(aq, sa, bq, sb)
    ah = _dequant_with_torch(aq, sa, 1, 128)
    assert np.array_equal(c, ah * 448.0 * 2.0 ** -7)
    # rank one: A = u 1^T (every row constant), B with columns of one value each
    u = torch.tensor([1.0, -2.0, 0.5]).view(3, 1).expand(3, 128).contiguous()
    v = torch.linspace(-1, 1, 128).view(1, 128).expand(128, 128).contiguous()
    aq, sa = oracle.quant_act_1x128(u.to(torch.bfloat16))
    bq, sb = oracle.quant_w_128x128(v.to(torch.bfloat16))
    c, _ = oracle.gemm_dequant(aq, sa, bq, sb)
    bcol = _dequant_with_torch(bq, sb, 128, 128)[0]
    arow = _dequant_with_torch(aq, sa, 1, 128)[:, 0]
    expect = arow[:, None] * 128 * bcol[None, :]
    assert np.allclose(c, expect, rtol=1e-12, atol=0)


def fgq_inputs_normal(shape, seed):
    import fgq_inputs
    return fgq_inputs.normal(shape, 1.0, seed)


def test_tolerance_check_detects_errors():
    c_ref = np.array([[1.0, -2.0]]); t = np.array([[10.0, 10.0]])
    ok, r = oracle.gemm_within_tolerance(c_ref + 0.019, c_ref, t)
    assert ok and r <= 2e-3
    ok, _ = oracle.gemm_within_tolerance(c_ref + 0.021, c_ref, t)
    assert not ok
    ok, _ = oracle.gemm_within_tolerance(np.array([[np.nan, -2.0]]), c_ref, t)
    assert not ok
    # bf16 output: the output rounding (2^-8 of the value) is added to the bound
    c_ref = np.array([[100.0]]); t = np.array([[100.0]])
    ok, _ = oracle.gemm_within_tolerance(c_ref + 0.2 + 0.39, c_ref, t, out_bf16=True)
    assert ok
    ok, _ = oracle.gemm_within_tolerance(c_ref + 0.2 + 0.41, c_ref, t, out_bf16=True)
    assert not ok
    ok, _ = oracle.gemm_within_tolerance(c_ref + 0.39, c_ref, t, out_bf16=False)
    assert not ok


# ---- MXFP4: E2M1 elements, UE8M0 scale per 32 ------------------------------

# The E2M1 values the page lists (§NVFP4 Two-Level Scaling).
E2M1_PAGE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_is_the_page_list():
    for c in range(8):
        assert oracle.e2m1_decode(c) == E2M1_PAGE[c]
        neg = oracle.e2m1_decode(c | 8)
        assert neg == -E2M1_PAGE[c] and math.copysign(1.0, neg) == -1.0


def test_e2m1_encode_nearest_even_saturating():
    for c in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_decode(c)) == c
    # brute-force nearest over a fine grid, ties to the even code
    vals = np.concatenate([np.linspace(-8, 8, 4097), [1e-30, -1e-30, 1e30, -1e30]])
    for v in vals:
        c = oracle.e2m1_encode(v)
        mag = abs(v)
        dists = [abs(e - min(mag, 6.0)) for e in E2M1_PAGE]
        best = min(dists)
        ties = [i for i, d in enumerate(dists) if d == best]
        want = ties[0] if len(ties) == 1 else [i for i in ties if i % 2 == 0][0]
        assert c & 7 == want, (v, c)
        if v < 0:
            assert c & 8
    for lo, hi in zip(range(7), range(1, 8)):  # every midpoint goes to the even code
        mid = (E2M1_PAGE[lo] + E2M1_PAGE[hi]) / 2
        assert oracle.e2m1_encode(mid) == (lo if lo % 2 == 0 else hi)


def test_mxfp4_scales_codes_and_packing():
    import fgq_inputs
    R, K = 64, 512
    x = fgq_inputs.exponent_spread((R, K), 40, 1, seed=9)
    x[3, 64:96] = 0.0                      # a zero group
    q, s = oracle.quant_mxfp4_1x32(x)
    assert q.shape == (R, K // 2) and s.shape == (R, K // 32)
    xf = x.float().numpy().astype(np.float64)
    dec = np.array([oracle.e2m1_decode(c) for c in range(16)])
    codes = np.stack([q & 15, q >> 4], axis=-1).reshape(R, K)   # element 2j = low nibble
    for r in range(R):
        for g in range(K // 32):
            grp = xf[r, 32 * g:32 * g + 32]
            amax = np.abs(grp).max()
            scale = 2.0 ** (int(s[r, g]) - 127)
            if amax == 0:
                assert s[r, g] == 127
            else:
                assert 3.0 < amax / scale <= 6.0   # power-of-two ceiling of amax / 6
            y = grp / scale
            got = dec[codes[r, 32 * g:32 * g + 32]]
            err = np.abs(got - y)
            nearest = np.min(np.abs(np.abs(y)[:, None] - np.array(E2M1_PAGE)[None, :]), axis=1)
            assert np.all(err <= nearest + 1e-300)  # every code is a nearest value


def test_mxfp4_gemm_matches_numpy_dequant():
    import fgq_inputs
    M, N, K = 24, 40, 256
    a = fgq_inputs.exponent_spread((M, K), 10, 1, seed=1)
    b = fgq_inputs.exponent_spread((N, K), 10, 1, seed=2)
    aq, sa = oracle.quant_mxfp4_1x32(a)
    bq, sb = oracle.quant_mxfp4_1x32(b)
    table = np.array(E2M1_PAGE + [-v for v in E2M1_PAGE])

    def deq(q, s):
        codes = np.stack([q & 15, q >> 4], axis=-1).reshape(q.shape[0], -1)
        return table[codes] * np.repeat(np.exp2(s.astype(np.float64) - 127.0), 32, axis=1)

    ah, bh = deq(aq, sa), deq(bq, sb)
    c, t = oracle.gemm_mxfp4(aq, sa, bq, sb)
    assert np.allclose(c, ah @ bh.T, rtol=0, atol=1e-12 * (np.abs(ah) @ np.abs(bh).T).max())
    assert np.allclose(t, np.abs(ah) @ np.abs(bh).T, rtol=1e-12)


# ---- NVFP4 (§NVFP4 Two-Level Scaling: global fp32 x E4M3 per 16 x E2M1) ----

def _bf16_row(vals):
    """A bf16 row from values that bf16 represents exactly."""
    t = torch.tensor(vals, dtype=torch.float32)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.float(), t)
    return b


def _nv_codes(q):
    return np.stack([q & 15, q >> 4], axis=-1).reshape(q.shape[0], -1)


def test_nvfp4_global_scale_closed_forms():
    # amax = 2688 * 2^k (2688 = 6 * 448 = 1.3125 * 2^11, exact in bf16) gives 2^k
    for k in (-20, -3, 0, 1, 7):
        amax = 2688.0 * 2.0 ** k
        x = _bf16_row([0.5 * amax, -amax, 0.25 * amax, 0.0]).reshape(2, 2)
        assert oracle.nvfp4_global_scale(x) == np.float32(2.0 ** k)
    assert oracle.nvfp4_global_scale(torch.zeros((3, 16), dtype=torch.bfloat16)) == 1.0
    neg0 = torch.full((2, 16), -0.0, dtype=torch.bfloat16)
    assert oracle.nvfp4_global_scale(neg0) == 1.0


def test_nvfp4_blocks_by_hand():
    """Blocks worked out by hand from the E4M3 and E2M1 definitions (g = 1)."""
    blk_a = [6, -6, 3, 1.5, 0.75, 0.25, -0.25, 5, 2.5, 1.25, 0.5, 4, 2, 1, 0, -0.0]
    # amax 6: t = 6/6 = 1 -> E4M3 0x38 (1.0), D = 1; 0.75, 0.25, 5, 2.5 and 1.25
    # are midpoints and go to the even code (1.0, 0, 4, 2, 1)
    want_a = [7, 15, 5, 3, 2, 0, 8, 6, 4, 2, 1, 6, 4, 2, 0, 8]
    # amax 6.375: t = 1.0625, the midpoint of 1.0 and 1.125 -> 1.0 (even);
    # 6.375 / 1 saturates to 6
    blk_b = [6.375, 1, -2, 0.5] + [0.0] * 12
    want_b = [7, 2, 12, 1] + [0] * 12
    # all zeros: t = 0 -> code 0, D = 0 -> signed zeros
    blk_c = [0.0, -0.0] * 8
    want_c = [0, 8] * 8
    # amax 12: t = 2 -> 0x40, D = 2: 12 -> 6, 3 -> 1.5, 1 -> 0.5, 0.5 -> 0.25 (tie -> 0)
    blk_d = [12, 3, 1, 0.5, -7, 9] + [0.0] * 10
    # -7 / 2 = -3.5, midpoint of 3 and 4 -> 4 (even code 6); 9 / 2 = 4.5 -> 4
    want_d = [7, 3, 1, 0, 14, 6] + [0] * 10
    x = _bf16_row(blk_a + blk_b + blk_c + blk_d).reshape(1, 64)
    q, s, g = oracle.quant_nvfp4_1x16(x, g=1.0)
    assert g == 1.0
    assert list(s[0]) == [0x38, 0x38, 0x00, 0x40]
    assert list(_nv_codes(q)[0]) == want_a + want_b + want_c + want_d
    assert q[0, 0] == (7 | (15 << 4))  # element 0 in the low nibble


def test_nvfp4_block_scale_under_a_global_scale():
    # tensor amax 336 = 2688 / 8 -> g = 0.125, 6 g = 0.75
    # block 0: amax 336 -> t = 448 -> 0x7E, D = 56: 336 -> 6, 28 -> 0.5
    # block 1: amax 21 -> t = 28 = 1.75 * 2^4 -> 0x5E, D = 3.5: 21 -> 6, 7 -> 2
    x = _bf16_row([336, 28] + [0.0] * 14 + [21, -7] + [0.0] * 14).reshape(1, 32)
    q, s, g = oracle.quant_nvfp4_1x16(x)
    assert g == np.float32(0.125)
    assert list(s[0]) == [0x7E, 0x5E]
    assert oracle.e4m3_decode(0x5E) == 28.0
    assert list(_nv_codes(q)[0][[0, 1, 16, 17]]) == [7, 1, 7, 12]


def test_nvfp4_block_maximum_maps_to_six():
    """With a normal E4M3 block scale s (within 2^-4 of t), the block's
    largest element lands in [6/(1+2^-4), 6/(1-2^-4)] in units of g s, which
    E2M1 rounds (or saturates) to 6."""
    import fgq_inputs
    x = fgq_inputs.exponent_spread((64, 512), 6, 1, seed=21)
    q, s, g = oracle.quant_nvfp4_1x16(x)
    codes = _nv_codes(q)
    xf = x.float().numpy()
    sdec = torch.from_numpy(s.copy()).view(torch.float8_e4m3fn).float().numpy()
    checked = 0
    for r in range(64):
        for b in range(32):
            blk = xf[r, 16 * b:16 * b + 16]
            if sdec[r, b] < 2.0 ** -6:   # subnormal block scale: wider rounding
                continue
            i = int(np.argmax(np.abs(blk)))
            assert codes[r, 16 * b + i] & 7 == 7
            assert (codes[r, 16 * b + i] >> 3) == (1 if blk[i] < 0 else 0)
            checked += 1
    assert checked > 1000


def test_nvfp4_gemm_matches_numpy_page_dequant():
    """C against numpy's matmul of operands decoded by the page's formula,
    global * float(block_scale) * e2m1, with torch's E4M3 decode."""
    import fgq_inputs
    M, N, K = 24, 40, 256
    a = fgq_inputs.exponent_spread((M, K), 8, 1, seed=3)
    b = fgq_inputs.exponent_spread((N, K), 8, 1, seed=4)
    aq, sa, ga = oracle.quant_nvfp4_1x16(a)
    bq, sb, gb = oracle.quant_nvfp4_1x16(b)
    table = np.array(E2M1_PAGE + [-v for v in E2M1_PAGE])

    def deq(q, s, g):
        blk = torch.from_numpy(s.copy()).view(torch.float8_e4m3fn).double().numpy()
        return float(g) * np.repeat(blk, 16, axis=1) * table[_nv_codes(q)]

    ah, bh = deq(aq, sa, ga), deq(bq, sb, gb)
    c, t = oracle.gemm_nvfp4(aq, sa, ga, bq, sb, gb)
    assert np.allclose(c, ah @ bh.T, rtol=0, atol=1e-12 * (np.abs(ah) @ np.abs(bh).T).max())
    assert np.allclose(t, np.abs(ah) @ np.abs(bh).T, rtol=1e-12)
    rows, cols = np.array([0, 5, 23]), np.array([39, 0, 17])
    c2, t2 = oracle.gemm_nvfp4_at(aq, sa, ga, bq, sb, gb, rows, cols)
    assert np.array_equal(c2, c[rows, cols]) and np.array_equal(t2, t[rows, cols])
    # and the dequantised values stay within one E2M1 step of the inputs
    af = a.float().numpy().astype(np.float64)
    d = np.repeat(float(ga) * torch.from_numpy(sa.copy()).view(torch.float8_e4m3fn).double().numpy(), 16, axis=1)
    assert np.all(np.abs(ah - af) <= 2.0 * d + 1e-300)


def test_parallel_gemm_reference_is_the_whole_matrix_call():
    """oracle.threads only slices the output by column blocks and runs the
    oracle on each slice: its (C, T) equal one whole-matrix call bit for
    bit, for any slice width and thread count."""
    from oracle.threads import gemm_dequant_parallel
    a = fgq_inputs.outlier((70, 384), 1e-2, 100.0, seed=21)
    b = fgq_inputs.exponent_spread((384, 640), 6, 128, seed=22)
    aq, sa = oracle.quant_act_1x128(a)
    bq, sb = oracle.quant_w_128x128(b)
    c, t = oracle.gemm_dequant(aq, sa, bq, sb)
    for workers, per in ((1, 1), (3, 1), (4, 2), (2, 5)):
        cp, tp = gemm_dequant_parallel(aq, sa, bq, sb, workers=workers, blocks_per_task=per)
        assert np.array_equal(cp.view(np.uint64), c.view(np.uint64))
        assert np.array_equal(tp.view(np.uint64), t.view(np.uint64))


def test_fp4_scale_tiles_by_hand():
    """Positions worked out by hand from the tiled layout's definition
    (512-byte tiles of 128 rows x 4 factor bytes; in a tile, row r at
    16 (r % 32) + 4 ((r % 128) / 32), factor byte f at + f % 4)."""
    R, F = 130, 8
    r = np.arange(R)[:, None]
    f = np.arange(F)[None, :]
    s = ((7 * r + 3 * f + 1) % 251).astype(np.uint8)
    t = oracle.fp4_scale_tiles(s)
    assert t.shape == (2 * 128 * F,)
    cases = {(0, 0): 0, (1, 0): 16, (32, 0): 4, (64, 4): 520, (33, 5): 533,
             (127, 3): 511, (129, 7): 1555, (128, 0): 1024, (96, 2): 14}
    for (rr, ff), off in cases.items():
        assert t[off] == s[rr, ff], (rr, ff, off)
    # rows 130..255 of the second row tile are padding: zero
    assert t[1024 + 2 * 16] == 0 and t[1024 + 31 * 16 + 3 * 4 + 3] == 0


def test_fp4_scale_tiles_is_a_permutation_matching_the_tensor_core_reading():
    """Every code lands exactly once, and read as [row tile, cell, lane i,
    quarter j, byte b] the tiles give code s[128 tile + 32 j + i, 4 cell + b]:
    the factor of row m sits in lane m % 32 of quarter m / 32."""
    R, F = 256, 12
    s = np.arange(R * F, dtype=np.int64).reshape(R, F)
    lo = (s % 256).astype(np.uint8)
    hi = (s // 256).astype(np.uint8)
    tl, th = oracle.fp4_scale_tiles(lo), oracle.fp4_scale_tiles(hi)
    back = tl.astype(np.int64) + 256 * th.astype(np.int64)
    assert np.array_equal(np.sort(back), np.arange(R * F))
    v = back.reshape(R // 128, F // 4, 32, 4, 4)
    for rb in range(R // 128):
        for c in range(F // 4):
            for i in (0, 5, 31):
                for j in range(4):
                    m = 128 * rb + 32 * j + i
                    assert list(v[rb, c, i, j]) == list(s[m, 4 * c:4 * c + 4])
    with pytest.raises(ValueError):
        oracle.fp4_scale_tiles(np.zeros((4, 6), dtype=np.uint8))
