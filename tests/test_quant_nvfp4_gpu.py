"""Parity of the NVFP4 quantizer (E2M1 elements, an E4M3 scale per 16 and an
fp32 per-tensor scale; "Fine-Grained FP8/FP4 Quantization", §NVFP4
Two-Level Scaling) with the oracle: the global scale, the codes and the
block-scale codes bit for bit."""
import numpy as np
import pytest
import torch

import fgq_inputs
import oracle

pytestmark = pytest.mark.gpu


def _dev(x_cpu, dev, pad):
    if not pad:
        return x_cpu.to(dev)
    R, K = x_cpu.shape
    big = torch.zeros((R, K + pad), dtype=torch.bfloat16)
    big[:, :K] = x_cpu
    return big.to(dev)[:, :K]


def _check(fgq, x_cpu, dev, pad=0):
    x = _dev(x_cpu, dev, pad)
    q, s, g = fgq.quant_nvfp4_1x16(x)
    torch.cuda.synchronize()
    go = oracle.nvfp4_global_scale(x_cpu)
    gg = g.cpu().numpy()[0]
    assert np.float32(gg).view(np.uint32) == np.float32(go).view(np.uint32), (gg, go)
    qo, so, _ = oracle.quant_nvfp4_1x16(x_cpu, g=go)
    sg, qg = s.cpu().numpy(), q.cpu().numpy()
    bad_s = np.argwhere(sg != so)
    assert bad_s.size == 0, f"{len(bad_s)} block-scale codes differ, first at {tuple(bad_s[0])}"
    bad = np.argwhere(qg != qo)
    assert bad.size == 0, (f"{len(bad)} code bytes differ, first at {tuple(bad[0])}: "
                           f"{qg[tuple(bad[0])]:#04x} vs {qo[tuple(bad[0])]:#04x}")


@pytest.mark.parametrize("R,K,pad", [(1, 16, 0), (7, 96, 8), (64, 1024, 0), (33, 7168, 64)])
def test_nvfp4_matches_oracle(fgq, cuda_dev, R, K, pad):
    x = fgq_inputs.outlier((R, K), 1e-2, 100.0, seed=R + K)
    _check(fgq, x, cuda_dev, pad)


def test_nvfp4_block_scales_across_binades(fgq, cuda_dev):
    """Blocks whose maxima fall 0 to 40 binades below the tensor maximum: E4M3
    block scales from 448 down through the subnormals to 0 (signed zeros)."""
    x = fgq_inputs.exponent_spread((256, 1024), 20, 1, seed=3)
    x[0, :16] = 0.0
    x[1, 16:32] = -0.0
    x[2, :] = torch.tensor(3.3e38, dtype=torch.bfloat16)  # near the bf16 maximum
    _check(fgq, x, cuda_dev)


def test_nvfp4_tiny_tensor(fgq, cuda_dev):
    """A tensor of bf16 subnormals: a subnormal global scale and products
    g * s near the bottom of fp32."""
    g = torch.Generator().manual_seed(5)
    bits = torch.randint(0, 0x80, (64, 256), generator=g, dtype=torch.int32)
    signs = torch.randint(0, 2, (64, 256), generator=g, dtype=torch.int32) << 15
    x = (bits | signs).to(torch.int16).view(torch.bfloat16)
    _check(fgq, x, cuda_dev)


def test_nvfp4_every_bf16_magnitude(fgq, cuda_dev):
    """Every finite bf16 value as an element of a block, under block maxima in
    several binades: each block is its maximum plus 15 values below it, in
    one tensor whose maximum sets g."""
    allbits = np.arange(0, 0x7F80, dtype=np.uint16)
    rows = []
    for amax_bits in (0x3F80, 0x3FC0, 0x0080, 0x0001, 0x7F7F, 0x2000, 0x5555):
        vals = allbits[allbits <= amax_bits]
        signs = np.where(np.arange(vals.size) % 2 == 0, 0, 0x8000).astype(np.uint16)
        vals = vals | signs
        n = (vals.size + 14) // 15
        vals = np.concatenate([vals, np.zeros(n * 15 - vals.size, np.uint16)]).reshape(n, 15)
        rows.append(np.concatenate([np.full((n, 1), amax_bits, np.uint16), vals], axis=1))
    blocks = np.concatenate(rows)
    B = blocks.shape[0] - blocks.shape[0] % 16
    x = torch.from_numpy(blocks[:B].reshape(-1, 256).view(np.int16)).view(torch.bfloat16)
    _check(fgq, x, cuda_dev)
    # and the same blocks under a global scale of 1 (every block scale saturates or not)
    q, s, _ = fgq.quant_nvfp4_1x16(x.to(cuda_dev), g=torch.ones(1, device=cuda_dev))
    qo, so, _ = oracle.quant_nvfp4_1x16(x, g=1.0)
    assert np.array_equal(s.cpu().numpy(), so) and np.array_equal(q.cpu().numpy(), qo)


def test_nvfp4_all_zero_tensor(fgq, cuda_dev):
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    x[1] = -0.0
    _check(fgq, x, cuda_dev)


def test_nvfp4_full_size(fgq, cuda_dev):
    x = fgq_inputs.student_t((4096, 7168), 3, 1.0, seed=6)
    _check(fgq, x, cuda_dev)


def _defined(R, F):
    """The bytes of the tiled layout that hold a code (not row padding)."""
    return oracle.fp4_scale_tiles(np.ones((R, F), np.uint8)) == 1


@pytest.mark.parametrize("R,K,pad", [(1, 64, 0), (7, 384, 8), (130, 1024, 0), (33, 7168, 64),
                                     (256, 192, 0)])
def test_nvfp4_tiled_scales_match_oracle(fgq, cuda_dev, R, K, pad):
    """The tiled-scale quantizer: global scale and codes as the row-major
    one, block scales bit for bit the oracle's in the tiled layout."""
    x_cpu = fgq_inputs.outlier((R, K), 1e-2, 100.0, seed=R + K + 2)
    x = _dev(x_cpu, cuda_dev, pad)
    q, t, g = fgq.quant_nvfp4_1x16_tiled(x)
    torch.cuda.synchronize()
    go = oracle.nvfp4_global_scale(x_cpu)
    assert np.float32(g.cpu().numpy()[0]).view(np.uint32) == np.float32(go).view(np.uint32)
    qo, so, _ = oracle.quant_nvfp4_1x16(x_cpu, g=go)
    mask = _defined(R, K // 16)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(t.cpu().numpy()[mask], oracle.fp4_scale_tiles(so)[mask])
    assert fgq.device_error() == 0
