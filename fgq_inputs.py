"""Seeded synthetic inputs for fine-grained FP8 quantization and GEMM.

This module draws random bf16 matrices and nothing else: it holds none of
the method's arithmetic (no scale, no encoding, no product).  It is the one
piece both the oracle-side tests and the GPU path use, so that both see the
same bf16 bits.

Distributions follow the workloads of the "Fine-Grained FP8/FP4
Quantization" page (§Scaling Granularities: an outlier ruins a per-tensor
scale; activations vary per channel):
  normal       N(0, std^2)
  student_t    t with nu degrees of freedom: z / sqrt(chi2_nu / nu), where
               chi2_nu is a sum of nu squared standard normals (heavy tails,
               the activation stand-in)
  outlier      N(0, 1) with a fraction of entries, at seeded uniform
               positions, multiplied by a factor
All are drawn in fp32 on the CPU with a seeded torch.Generator and rounded
to bf16 (round to nearest even).
"""
from __future__ import annotations

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float = 1.0, seed: int = 0) -> torch.Tensor:
    g = _gen(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def student_t(shape, nu: int = 3, scale: float = 1.0, seed: int = 0) -> torch.Tensor:
    g = _gen(seed)
    z = torch.randn(*shape, generator=g, dtype=torch.float32)
    chi2 = torch.zeros(*shape, dtype=torch.float32)
    for _ in range(int(nu)):
        e = torch.randn(*shape, generator=g, dtype=torch.float32)
        chi2.addcmul_(e, e)
    x = z.div_(torch.sqrt(chi2.div_(float(nu))))
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def outlier(shape, frac: float = 1e-3, factor: float = 100.0, seed: int = 0) -> torch.Tensor:
    g = _gen(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    n = x.numel()
    count = int(round(frac * n))
    pos = torch.randperm(n, generator=g)[:count]
    flat = x.view(-1)
    flat[pos] *= factor
    return x.to(torch.bfloat16)


def exponent_spread(shape, spread: int, block_rows: int, seed: int = 0) -> torch.Tensor:
    """N(0, 1) values, each block of block_rows x 128 entries multiplied by
    2^e with e uniform in [-spread, spread] (exact in bf16): block_rows = 1
    gives activation-like 1x128 groups of very different magnitudes,
    block_rows = 128 the same for 128x128 weight blocks."""
    g = _gen(seed)
    rows, cols = shape
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    br = (rows + block_rows - 1) // block_rows
    bc = (cols + 127) // 128
    e = torch.randint(-spread, spread + 1, (br, bc), generator=g).to(torch.float32)
    f = torch.exp2(e).repeat_interleave(block_rows, 0)[:rows].repeat_interleave(128, 1)[:, :cols]
    return (x * f).to(torch.bfloat16)


# Named workloads with their shapes and distributions.  Seeds are fixed so a
# run on any machine regenerates the same bits.
def tiny(seed: int = 0):
    """A bf16 [128, 256], B bf16 [256, 128], N(0, 1)."""
    return normal((128, 256), 1.0, seed), normal((256, 128), 1.0, seed + 1)


def outlier_gemm(n: int = 1024, seed: int = 0):
    """A, B bf16 [n, n], N(0, 1) with 0.1% of entries multiplied by 100."""
    return outlier((n, n), 1e-3, 100.0, seed), outlier((n, n), 1e-3, 100.0, seed + 1)


def quant_bw(seed: int = 0, m: int = 16384, k: int = 7168, n: int = 7168):
    """Activations [m, k] Student-t (nu = 3), weight [k, n] N(0, 0.02^2)."""
    return student_t((m, k), 3, 1.0, seed), normal((k, n), 0.02, seed + 1)


def large_prefill(seed: int = 0, m: int = 4096, k: int = 7168, n: int = 7168):
    """A [m, k] N(0, 1), B [k, n] N(0, 0.02^2)."""
    return normal((m, k), 1.0, seed), normal((k, n), 0.02, seed + 1)


def skinny(m: int, seed: int = 0, n: int = 24576, k: int = 1536):
    """A [m, k] N(0, 1), B [k, n] N(0, 0.02^2), m in {16, 64, 256}."""
    return normal((m, k), 1.0, seed), normal((k, n), 0.02, seed + 1)
