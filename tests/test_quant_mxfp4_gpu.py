"""Parity of the MXFP4 quantizer (E2M1 elements, one UE8M0 scale per 32;
"Fine-Grained FP8/FP4 Quantization", §UE8M0 vs E4M3 Scale Formats) with the
oracle: codes and scale codes bit for bit."""
import numpy as np
import pytest
import torch

import fgq_inputs
import oracle

pytestmark = pytest.mark.gpu


def _check(fgq, x_cpu, dev, pad=0):
    R, K = x_cpu.shape
    if pad:
        big = torch.zeros((R, K + pad), dtype=torch.bfloat16)
        big[:, :K] = x_cpu
        x = big.to(dev)[:, :K]
    else:
        x = x_cpu.to(dev)
    q, s = fgq.quant_mxfp4_1x32(x)
    torch.cuda.synchronize()
    qo, so = oracle.quant_mxfp4_1x32(x_cpu)
    sg, qg = s.cpu().numpy(), q.cpu().numpy()
    bad_s = np.argwhere(sg != so)
    assert bad_s.size == 0, f"{len(bad_s)} scale codes differ, first at {tuple(bad_s[0])}"
    bad = np.argwhere(qg != qo)
    assert bad.size == 0, (f"{len(bad)} code bytes differ, first at {tuple(bad[0])}: "
                           f"{qg[tuple(bad[0])]:#04x} vs {qo[tuple(bad[0])]:#04x}")


@pytest.mark.parametrize("R,K,pad", [(1, 32, 0), (7, 96, 8), (64, 1024, 0), (33, 7168, 64)])
def test_mxfp4_matches_oracle(fgq, cuda_dev, R, K, pad):
    x = fgq_inputs.outlier((R, K), 1e-2, 100.0, seed=R + K)
    _check(fgq, x, cuda_dev, pad)


def test_mxfp4_scales_across_binades_zero_groups(fgq, cuda_dev):
    """Group maxima over 250 binades (down to the 2^-127 clamp and up to the
    largest bf16 values), zero groups and groups of negative zeros."""
    x = fgq_inputs.exponent_spread((256, 1024), 125, 1, seed=3)
    x[0, :32] = 0.0
    x[1, 32:64] = -0.0
    x[2, :] = torch.tensor(3.3e38, dtype=torch.bfloat16)  # near the bf16 maximum
    _check(fgq, x, cuda_dev)


def test_mxfp4_every_bf16_magnitude(fgq, cuda_dev):
    """Every finite bf16 value as an element of a group, under group maxima in
    several binades: each group is its maximum plus 31 values below it."""
    allbits = np.arange(0, 0x7F80, dtype=np.uint16)          # finite non-negative patterns
    rows = []
    for amax_bits in (0x3F80, 0x3FC0, 0x0080, 0x0001, 0x7F7F, 0x2000, 0x5555):
        vals = allbits[allbits <= amax_bits]
        signs = np.where(np.arange(vals.size) % 2 == 0, 0, 0x8000).astype(np.uint16)
        vals = vals | signs
        n = (vals.size + 30) // 31
        vals = np.concatenate([vals, np.zeros(n * 31 - vals.size, np.uint16)]).reshape(n, 31)
        grp = np.concatenate([np.full((n, 1), amax_bits, np.uint16), vals], axis=1)  # [n, 32]
        rows.append(grp)
    groups = np.concatenate(rows)                            # [G, 32]
    G = groups.shape[0] - groups.shape[0] % 8
    x = torch.from_numpy(groups[:G].reshape(-1, 256).view(np.int16)).view(torch.bfloat16)
    _check(fgq, x, cuda_dev)


def test_mxfp4_full_size(fgq, cuda_dev):
    x = fgq_inputs.student_t((4096, 7168), 3, 1.0, seed=6)
    _check(fgq, x, cuda_dev)


def _defined(R, F):
    """The bytes of the tiled layout that hold a code (not row padding)."""
    return oracle.fp4_scale_tiles(np.ones((R, F), np.uint8)) == 1


@pytest.mark.parametrize("R,K,pad", [(1, 128, 0), (7, 384, 8), (130, 1024, 0), (33, 7168, 64),
                                     (256, 256, 0)])
def test_mxfp4_tiled_scales_match_oracle(fgq, cuda_dev, R, K, pad):
    """The tiled-scale quantizer: codes as the row-major one, scales bit for
    bit the oracle's scales in the tiled layout; and the relayout of the
    row-major scales gives the same tiles."""
    x_cpu = fgq_inputs.outlier((R, K), 1e-2, 100.0, seed=R + K + 1)
    if pad:
        big = torch.zeros((R, K + pad), dtype=torch.bfloat16)
        big[:, :K] = x_cpu
        x = big.to(cuda_dev)[:, :K]
    else:
        x = x_cpu.to(cuda_dev)
    q, t = fgq.quant_mxfp4_1x32_tiled(x)
    q2, s2 = fgq.quant_mxfp4_1x32(x)
    t2 = fgq.fp4_scales_to_tiles(s2)
    torch.cuda.synchronize()
    qo, so = oracle.quant_mxfp4_1x32(x_cpu)
    to = oracle.fp4_scale_tiles(so)
    mask = _defined(R, K // 32)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(t.cpu().numpy()[mask], to[mask])
    assert np.array_equal(t2.cpu().numpy()[mask], to[mask])
    assert fgq.device_error() == 0


@pytest.mark.parametrize("R,F", [(1, 4), (129, 8), (300, 12), (4096, 224)])
def test_fp4_scales_to_tiles_matches_oracle(fgq, cuda_dev, R, F):
    s = np.random.default_rng(R * F).integers(0, 256, (R, F), dtype=np.uint8)
    t = fgq.fp4_scales_to_tiles(torch.from_numpy(s).to(cuda_dev))
    torch.cuda.synchronize()
    assert t.numel() == fgq.fp4_scale_tiles_bytes(R, F) == ((R + 127) // 128) * 128 * F
    mask = _defined(R, F)
    assert np.array_equal(t.cpu().numpy()[mask], oracle.fp4_scale_tiles(s)[mask])


def test_mxfp4_tiled_codes_at_a_4_byte_offset(fgq, cuda_dev):
    """Codes written to a buffer only 4-byte aligned (the API's minimum)
    equal those written to a 16-byte-aligned one, and so do the scale
    tiles."""
    R, K = 33, 384
    x = fgq_inputs.outlier((R, K), 1e-2, 100.0, seed=91).to(cuda_dev)
    q, t = fgq.quant_mxfp4_1x32_tiled(x)
    buf = torch.full((R * K // 2 + 16,), 0xAB, dtype=torch.uint8, device=cuda_dev)
    xq_off = buf[4:4 + R * K // 2].view(R, K // 2)
    assert xq_off.data_ptr() % 16 == 4
    q2, t2 = fgq.quant_mxfp4_1x32_tiled(x, xq=xq_off)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(t, t2)
    # nothing written outside the codes
    assert bool((buf[:4] == 0xAB).all()) and bool((buf[4 + R * K // 2:] == 0xAB).all())
