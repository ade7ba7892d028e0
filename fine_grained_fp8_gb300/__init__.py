"""Fine-grained FP8 quantization and block-scaled FP8 GEMM for GB300 (sm_103a).

Tensor-level wrappers over the C ABI of libfgq.so (include/fgq.h).  PyTorch
provides device memory and the current CUDA stream; all arithmetic runs in
the library's kernels:

  quant_act_1x128(x)        bf16 [M, K] -> (E4M3 codes [M, K] uint8, fp32 [M, K/128])
  quant_act_128x1(x)        bf16 [M, K] -> (E4M3 codes [K, M] uint8, fp32 [K, M/128]),
                            groups of 128 rows (for a GEMM reducing over M)
  quant_w_128x128(w)        bf16 [K, N] -> (E4M3 codes [N, K] uint8 (K-major),
                                            fp32 [K/128, N/128])
  quant_operands(x, w)      both of the above in one launch
  gemm_fp8_blockscaled(aq, sa, bq, sb, out_dtype)
                            C [M, N] = sum over 128-wide K chunks of
                            (Aq Bq)_chunk * sa * sb

("Fine-Grained FP8/FP4 Quantization": §Scaling Granularities, §DeepGEMM.)
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import (FGQ_OUT_BF16, FGQ_OUT_F32, FGQ_SCALE_FP32, FGQ_SCALE_UE8M0, FgqError,
                   check, load)

__all__ = ["quant_act_1x128", "quant_act_128x1", "quant_operands", "quant_mxfp4_1x32", "nvfp4_global_scale",
           "quant_nvfp4_1x16", "quant_w_128x128", "gemm_fp8_blockscaled",
           "gemm_fp8_blockscaled_splitk", "gemm_fp8_blockscaled_fused_act", "gemm_mxfp4",
           "gemm_nvfp4", "fp4_scale_tiles_bytes", "fp4_scales_to_tiles",
           "quant_mxfp4_1x32_tiled", "quant_nvfp4_1x16_tiled", "gemm_mxfp4_tiled",
           "gemm_nvfp4_tiled", "ue8m0_scale_tiles_bytes", "ue8m0_scale_tiles",
           "gemm_fp8_ue8m0_tiled", "quant_operands_ue8m0_tiles", "splitk_workspace",
           "device_error",
           "FgqError", "load", "FGQ_SCALE_FP32", "FGQ_SCALE_UE8M0", "FGQ_OUT_F32",
           "FGQ_OUT_BF16", "scale_mode"]


def scale_mode(mode) -> int:
    if mode in ("fp32", FGQ_SCALE_FP32, None):
        return FGQ_SCALE_FP32
    if mode in ("ue8m0", FGQ_SCALE_UE8M0):
        return FGQ_SCALE_UE8M0
    raise ValueError(f"unknown scale mode {mode!r} (use 'fp32' or 'ue8m0')")


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _need_cuda(name: str, t: torch.Tensor, dtype) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def quant_act_1x128(x: torch.Tensor, mode="fp32", xq: torch.Tensor | None = None,
                    sx: torch.Tensor | None = None):
    """1x128 tile-wise quantization of bf16 activations x [M, K] (rows may be
    strided; the last dimension must be contiguous)."""
    _need_cuda("x", x, torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with a contiguous last dimension")
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((M, K // 128), dtype=torch.float32, device=x.device)
    _need_cuda("xq", xq, torch.uint8)
    _need_cuda("sx", sx, torch.float32)
    if xq.shape != (M, K) or xq.stride(1) != 1 or sx.shape != (M, K // 128) or not sx.is_contiguous():
        raise ValueError("xq must be [M, K] (contiguous rows) and sx a dense [M, K/128]")
    st = _lib.fgq_quant_act_1x128(x.data_ptr(), M, K, x.stride(0), xq.data_ptr(), xq.stride(0),
                                  sx.data_ptr(), scale_mode(mode), _stream(x))
    check("fgq_quant_act_1x128", st)
    return xq, sx


def quant_act_128x1(x: torch.Tensor, mode="fp32", xqt: torch.Tensor | None = None,
                    sxt: torch.Tensor | None = None):
    """128x1 (transposed) quantization of bf16 activations x [M, K] (rows may
    be strided): groups of 128 rows of one column.  Returns xqt [K, M] E4M3
    codes and sxt [K, M/128] scales, the A operand of a GEMM reducing over M
    (the same result as quant_act_1x128(x.t()))."""
    _need_cuda("x", x, torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with a contiguous last dimension")
    M, K = x.shape
    if xqt is None:
        xqt = torch.empty((K, M), dtype=torch.uint8, device=x.device)
    if sxt is None:
        sxt = torch.empty((K, M // 128), dtype=torch.float32, device=x.device)
    _need_cuda("xqt", xqt, torch.uint8)
    _need_cuda("sxt", sxt, torch.float32)
    if xqt.shape != (K, M) or not xqt.is_contiguous() or sxt.shape != (K, M // 128) \
            or not sxt.is_contiguous():
        raise ValueError("xqt must be a dense [K, M] and sxt a dense [K, M/128]")
    st = _lib.fgq_quant_act_128x1(x.data_ptr(), M, K, x.stride(0), xqt.data_ptr(), sxt.data_ptr(),
                                  scale_mode(mode), _stream(x))
    check("fgq_quant_act_128x1", st)
    return xqt, sxt


def quant_mxfp4_1x32(x: torch.Tensor, xq: torch.Tensor | None = None,
                     sx: torch.Tensor | None = None):
    """MXFP4 quantization of the rows of bf16 x [R, K]: E2M1 codes packed two
    per byte, xq [R, K/2] uint8 (even element in the low nibble), and one
    UE8M0 scale code per 32 elements, sx [R, K/32] uint8."""
    _need_cuda("x", x, torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with a contiguous last dimension")
    R, K = x.shape
    if xq is None:
        xq = torch.empty((R, K // 2), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((R, K // 32), dtype=torch.uint8, device=x.device)
    _need_cuda("xq", xq, torch.uint8)
    _need_cuda("sx", sx, torch.uint8)
    if xq.shape != (R, K // 2) or not xq.is_contiguous() or sx.shape != (R, K // 32) \
            or not sx.is_contiguous():
        raise ValueError("xq must be a dense [R, K/2] and sx a dense [R, K/32]")
    st = _lib.fgq_quant_mxfp4_1x32(x.data_ptr(), R, K, x.stride(0), xq.data_ptr(), sx.data_ptr(),
                                   _stream(x))
    check("fgq_quant_mxfp4_1x32", st)
    return xq, sx


def nvfp4_global_scale(x: torch.Tensor, g: torch.Tensor | None = None) -> torch.Tensor:
    """NVFP4 per-tensor scale of bf16 x [R, K] (amax / 2688, 1 for all zeros)
    as a one-element fp32 device tensor."""
    _need_cuda("x", x, torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with a contiguous last dimension")
    R, K = x.shape
    if g is None:
        g = torch.empty((1,), dtype=torch.float32, device=x.device)
    _need_cuda("g", g, torch.float32)
    st = _lib.fgq_nvfp4_global_scale(x.data_ptr(), R, K, x.stride(0), g.data_ptr(), _stream(x))
    check("fgq_nvfp4_global_scale", st)
    return g


def quant_nvfp4_1x16(x: torch.Tensor, g: torch.Tensor | None = None,
                     xq: torch.Tensor | None = None, sx: torch.Tensor | None = None):
    """NVFP4 quantization of the rows of bf16 x [R, K] under the global scale
    g (a one-element fp32 device tensor; computed with nvfp4_global_scale when
    None): E2M1 codes xq [R, K/2] uint8 (even element in the low nibble) and
    one E4M3 block-scale code per 16 elements, sx [R, K/16] uint8.  Returns
    (xq, sx, g)."""
    _need_cuda("x", x, torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with a contiguous last dimension")
    R, K = x.shape
    if g is None:
        g = nvfp4_global_scale(x)
    _need_cuda("g", g, torch.float32)
    if xq is None:
        xq = torch.empty((R, K // 2), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((R, K // 16), dtype=torch.uint8, device=x.device)
    _need_cuda("xq", xq, torch.uint8)
    _need_cuda("sx", sx, torch.uint8)
    if xq.shape != (R, K // 2) or not xq.is_contiguous() or sx.shape != (R, K // 16) \
            or not sx.is_contiguous():
        raise ValueError("xq must be a dense [R, K/2] and sx a dense [R, K/16]")
    st = _lib.fgq_quant_nvfp4_1x16(x.data_ptr(), R, K, x.stride(0), g.data_ptr(), xq.data_ptr(),
                                   sx.data_ptr(), _stream(x))
    check("fgq_quant_nvfp4_1x16", st)
    return xq, sx, g


def quant_w_128x128(w: torch.Tensor, mode="fp32", wq: torch.Tensor | None = None,
                    sw: torch.Tensor | None = None):
    """128x128 block-wise quantization of a bf16 weight w [K, N].  Returns the
    codes TRANSPOSED, wq [N, K] (K-major), and sw [K/128, N/128]."""
    _need_cuda("w", w, torch.bfloat16)
    if w.dim() != 2 or w.stride(1) != 1:
        raise ValueError("w must be 2-D with a contiguous last dimension")
    K, N = w.shape
    if wq is None:
        wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if sw is None:
        sw = torch.empty((K // 128, N // 128), dtype=torch.float32, device=w.device)
    _need_cuda("wq", wq, torch.uint8)
    _need_cuda("sw", sw, torch.float32)
    if wq.shape != (N, K) or not wq.is_contiguous() or sw.shape != (K // 128, N // 128) \
            or not sw.is_contiguous():
        raise ValueError("wq must be a dense [N, K] and sw a dense [K/128, N/128]")
    st = _lib.fgq_quant_w_128x128(w.data_ptr(), K, N, w.stride(0), wq.data_ptr(), sw.data_ptr(),
                                  scale_mode(mode), _stream(w))
    check("fgq_quant_w_128x128", st)
    return wq, sw


def quant_operands(x: torch.Tensor, w: torch.Tensor, mode="fp32", xq: torch.Tensor | None = None,
                   sx: torch.Tensor | None = None, wq: torch.Tensor | None = None,
                   sw: torch.Tensor | None = None):
    """Both GEMM operands in one launch: quant_act_1x128(x) and
    quant_w_128x128(w), bit for bit.  Returns (xq, sx, wq, sw)."""
    _need_cuda("x", x, torch.bfloat16)
    _need_cuda("w", w, torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1 or w.dim() != 2 or w.stride(1) != 1:
        raise ValueError("x and w must be 2-D with a contiguous last dimension")
    M, K = x.shape
    K2, N = w.shape
    if K2 != K:
        raise ValueError(f"x is [M, {K}] but w is [{K2}, N]")
    if x.device != w.device:
        raise ValueError("x and w must be on the same device")
    dev = x.device
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev) if xq is None else xq
    sx = torch.empty((M, K // 128), dtype=torch.float32, device=dev) if sx is None else sx
    wq = torch.empty((N, K), dtype=torch.uint8, device=dev) if wq is None else wq
    sw = torch.empty((K // 128, N // 128), dtype=torch.float32, device=dev) if sw is None else sw
    for name, t, dt in (("xq", xq, torch.uint8), ("sx", sx, torch.float32), ("wq", wq, torch.uint8),
                        ("sw", sw, torch.float32)):
        _need_cuda(name, t, dt)
    if xq.shape != (M, K) or xq.stride(1) != 1 or sx.shape != (M, K // 128) or not sx.is_contiguous():
        raise ValueError("xq must be [M, K] (contiguous rows) and sx a dense [M, K/128]")
    if wq.shape != (N, K) or not wq.is_contiguous() or sw.shape != (K // 128, N // 128) \
            or not sw.is_contiguous():
        raise ValueError("wq must be a dense [N, K] and sw a dense [K/128, N/128]")
    st = _lib.fgq_quant_operands(x.data_ptr(), M, K, x.stride(0), xq.data_ptr(), xq.stride(0),
                                 sx.data_ptr(), w.data_ptr(), N, w.stride(0), wq.data_ptr(),
                                 sw.data_ptr(), scale_mode(mode), _stream(x))
    check("fgq_quant_operands", st)
    return xq, sx, wq, sw


def gemm_fp8_blockscaled(aq: torch.Tensor, sa: torch.Tensor, bq: torch.Tensor,
                         sb: torch.Tensor, out_dtype=torch.float32, mode="fp32",
                         out: torch.Tensor | None = None) -> torch.Tensor:
    """C [M, N] = block-scaled FP8 product of aq [M, K] (1x128 scales sa) and the
    K-major weight codes bq [N, K] (128x128 scales sb [K/128, N/128])."""
    _need_cuda("aq", aq, torch.uint8)
    _need_cuda("bq", bq, torch.uint8)
    _need_cuda("sa", sa, torch.float32)
    _need_cuda("sb", sb, torch.float32)
    for name, t in (("aq", aq), ("bq", bq), ("sa", sa), ("sb", sb)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    M, K = aq.shape
    N, K2 = bq.shape
    if K2 != K or sa.shape != (M, K // 128) or sb.shape != (K // 128, N // 128):
        raise ValueError("shape mismatch: aq [M,K], sa [M,K/128], bq [N,K], sb [K/128,N/128]")
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=aq.device)
    _need_cuda("out", out, out_dtype)
    if out.shape != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] with contiguous rows")
    st = _lib.fgq_gemm_fp8_blockscaled_ex(
        aq.data_ptr(), sa.data_ptr(), bq.data_ptr(), sb.data_ptr(), out.data_ptr(), out.stride(0),
        M, N, K, FGQ_OUT_BF16 if out_dtype == torch.bfloat16 else FGQ_OUT_F32, scale_mode(mode),
        _stream(aq))
    check("fgq_gemm_fp8_blockscaled_ex", st)
    return out


def gemm_fp8_blockscaled_fused_act(a: torch.Tensor, bq: torch.Tensor, sb: torch.Tensor,
                                   out_dtype=torch.float32, mode="fp32",
                                   out: torch.Tensor | None = None) -> torch.Tensor:
    """C [M, N] for bf16 activations a [M, K] (rows may be strided), quantized
    1x128 inside the GEMM (same codes as quant_act_1x128), times the weight
    codes bq [N, K] with scales sb [K/128, N/128].  M <= 32 and A small
    enough to stay on chip (see include/fgq.h)."""
    _need_cuda("a", a, torch.bfloat16)
    _need_cuda("bq", bq, torch.uint8)
    _need_cuda("sb", sb, torch.float32)
    if a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a must be 2-D with a contiguous last dimension")
    if not bq.is_contiguous() or not sb.is_contiguous():
        raise ValueError("bq and sb must be contiguous")
    M, K = a.shape
    N, K2 = bq.shape
    if K2 != K or sb.shape != (K // 128, N // 128):
        raise ValueError("shape mismatch: a [M,K], bq [N,K], sb [K/128,N/128]")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    _need_cuda("out", out, out_dtype)
    if out.shape != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] with contiguous rows")
    st = _lib.fgq_gemm_fp8_blockscaled_fused_act(
        a.data_ptr(), a.stride(0), bq.data_ptr(), sb.data_ptr(), out.data_ptr(), out.stride(0),
        M, N, K, FGQ_OUT_BF16 if out_dtype == torch.bfloat16 else FGQ_OUT_F32, scale_mode(mode),
        _stream(a))
    check("fgq_gemm_fp8_blockscaled_fused_act", st)
    return out


def gemm_mxfp4(aq: torch.Tensor, sa: torch.Tensor, bq: torch.Tensor, sb: torch.Tensor,
               out_dtype=torch.float32, out: torch.Tensor | None = None) -> torch.Tensor:
    """C [M, N] from MXFP4 operands as quant_mxfp4_1x32 writes them: aq [M, K/2]
    and sa [M, K/32], bq [N, K/2] and sb [N, K/32] (the weight quantized as
    its transpose)."""
    for name, t in (("aq", aq), ("sa", sa), ("bq", bq), ("sb", sb)):
        _need_cuda(name, t, torch.uint8)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    M, K = aq.shape[0], 2 * aq.shape[1]
    N = bq.shape[0]
    if bq.shape != (N, K // 2) or sa.shape != (M, K // 32) or sb.shape != (N, K // 32):
        raise ValueError("shape mismatch: aq [M,K/2], sa [M,K/32], bq [N,K/2], sb [N,K/32]")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=aq.device)
    _need_cuda("out", out, out_dtype)
    if out.shape != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] with contiguous rows")
    st = _lib.fgq_gemm_mxfp4(aq.data_ptr(), sa.data_ptr(), bq.data_ptr(), sb.data_ptr(),
                             out.data_ptr(), out.stride(0), M, N, K,
                             FGQ_OUT_BF16 if out_dtype == torch.bfloat16 else FGQ_OUT_F32,
                             _stream(aq))
    check("fgq_gemm_mxfp4", st)
    return out


def gemm_nvfp4(aq: torch.Tensor, sa: torch.Tensor, ga: torch.Tensor, bq: torch.Tensor,
               sb: torch.Tensor, gb: torch.Tensor, out_dtype=torch.float32,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """C [M, N] from NVFP4 operands as quant_nvfp4_1x16 writes them: aq [M, K/2],
    sa [M, K/16] and the global scale ga; bq [N, K/2], sb [N, K/16] and gb
    (the weight quantized as its transpose)."""
    for name, t in (("aq", aq), ("sa", sa), ("bq", bq), ("sb", sb)):
        _need_cuda(name, t, torch.uint8)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    _need_cuda("ga", ga, torch.float32)
    _need_cuda("gb", gb, torch.float32)
    M, K = aq.shape[0], 2 * aq.shape[1]
    N = bq.shape[0]
    if bq.shape != (N, K // 2) or sa.shape != (M, K // 16) or sb.shape != (N, K // 16):
        raise ValueError("shape mismatch: aq [M,K/2], sa [M,K/16], bq [N,K/2], sb [N,K/16]")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=aq.device)
    _need_cuda("out", out, out_dtype)
    if out.shape != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] with contiguous rows")
    st = _lib.fgq_gemm_nvfp4(aq.data_ptr(), sa.data_ptr(), ga.data_ptr(), bq.data_ptr(),
                             sb.data_ptr(), gb.data_ptr(), out.data_ptr(), out.stride(0), M, N, K,
                             FGQ_OUT_BF16 if out_dtype == torch.bfloat16 else FGQ_OUT_F32,
                             _stream(aq))
    check("fgq_gemm_nvfp4", st)
    return out


def fp4_scale_tiles_bytes(R: int, F: int) -> int:
    """Bytes of FP4 block scales for R rows of F factor bytes (F = K/32 for
    MXFP4, K/16 for NVFP4) in the tiled layout: ceil(R/128) * 128 * F."""
    st, n = _lib.fgq_fp4_scale_tiles_bytes(R, F)
    check("fgq_fp4_scale_tiles_bytes", st)
    return n


def fp4_scales_to_tiles(s: torch.Tensor, tiles: torch.Tensor | None = None) -> torch.Tensor:
    """Row-major FP4 block scales s [R, F] uint8 (F % 4 == 0) in the tiled
    layout the _tiled GEMMs take: a 1-D uint8 tensor of
    fp4_scale_tiles_bytes(R, F) bytes (pad rows written as zeros)."""
    _need_cuda("s", s, torch.uint8)
    if s.dim() != 2 or not s.is_contiguous():
        raise ValueError("s must be a dense [R, F]")
    R, F = s.shape
    n = fp4_scale_tiles_bytes(R, F)
    if tiles is None:
        tiles = torch.empty((n,), dtype=torch.uint8, device=s.device)
    _need_cuda("tiles", tiles, torch.uint8)
    if tiles.numel() != n or not tiles.is_contiguous():
        raise ValueError(f"tiles must be a dense uint8 tensor of {n} bytes")
    st = _lib.fgq_fp4_scales_to_tiles(s.data_ptr(), R, F, tiles.data_ptr(), _stream(s))
    check("fgq_fp4_scales_to_tiles", st)
    return tiles


def _tiles_out(t, n, dev, name):
    if t is None:
        t = torch.empty((n,), dtype=torch.uint8, device=dev)
    _need_cuda(name, t, torch.uint8)
    if t.numel() != n or not t.is_contiguous():
        raise ValueError(f"{name} must be a dense uint8 tensor of {n} bytes")
    return t


def quant_mxfp4_1x32_tiled(x: torch.Tensor, xq: torch.Tensor | None = None,
                           s_tiles: torch.Tensor | None = None):
    """quant_mxfp4_1x32 with the scales in the tiled layout: returns (xq
    [R, K/2], scale tiles as a 1-D uint8 tensor).  K % 128 == 0."""
    _need_cuda("x", x, torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with a contiguous last dimension")
    R, K = x.shape
    if xq is None:
        xq = torch.empty((R, K // 2), dtype=torch.uint8, device=x.device)
    _need_cuda("xq", xq, torch.uint8)
    if xq.shape != (R, K // 2) or not xq.is_contiguous():
        raise ValueError("xq must be a dense [R, K/2]")
    tiles = _tiles_out(s_tiles, fp4_scale_tiles_bytes(R, K // 32), x.device, "s_tiles")
    st = _lib.fgq_quant_mxfp4_1x32_tiled(x.data_ptr(), R, K, x.stride(0), xq.data_ptr(),
                                         tiles.data_ptr(), _stream(x))
    check("fgq_quant_mxfp4_1x32_tiled", st)
    return xq, tiles


def quant_nvfp4_1x16_tiled(x: torch.Tensor, g: torch.Tensor | None = None,
                           xq: torch.Tensor | None = None, s_tiles: torch.Tensor | None = None):
    """quant_nvfp4_1x16 with the scales in the tiled layout: returns (xq
    [R, K/2], scale tiles as a 1-D uint8 tensor, g).  K % 64 == 0."""
    _need_cuda("x", x, torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with a contiguous last dimension")
    R, K = x.shape
    if g is None:
        g = nvfp4_global_scale(x)
    _need_cuda("g", g, torch.float32)
    if xq is None:
        xq = torch.empty((R, K // 2), dtype=torch.uint8, device=x.device)
    _need_cuda("xq", xq, torch.uint8)
    if xq.shape != (R, K // 2) or not xq.is_contiguous():
        raise ValueError("xq must be a dense [R, K/2]")
    tiles = _tiles_out(s_tiles, fp4_scale_tiles_bytes(R, K // 16), x.device, "s_tiles")
    st = _lib.fgq_quant_nvfp4_1x16_tiled(x.data_ptr(), R, K, x.stride(0), g.data_ptr(),
                                         xq.data_ptr(), tiles.data_ptr(), _stream(x))
    check("fgq_quant_nvfp4_1x16_tiled", st)
    return xq, tiles, g


def _fp4_tiled_operands(aq, sa, bq, sb, per):
    for name, t in (("aq", aq), ("sa", sa), ("bq", bq), ("sb", sb)):
        _need_cuda(name, t, torch.uint8)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    M, K = aq.shape[0], 2 * aq.shape[1]
    N = bq.shape[0]
    if bq.shape != (N, K // 2):
        raise ValueError("shape mismatch: aq [M, K/2], bq [N, K/2]")
    if K % per != 0 or (K // per) % 4 != 0:
        raise ValueError("K must give a whole number of 4-byte factor cells")
    if sa.numel() != fp4_scale_tiles_bytes(M, K // per) or \
            sb.numel() != fp4_scale_tiles_bytes(N, K // per):
        raise ValueError("sa / sb must be scale tiles of fp4_scale_tiles_bytes(rows, K/%d)" % per)
    return M, N, K


def gemm_mxfp4_tiled(aq: torch.Tensor, sa: torch.Tensor, bq: torch.Tensor, sb: torch.Tensor,
                     out_dtype=torch.float32, out: torch.Tensor | None = None) -> torch.Tensor:
    """gemm_mxfp4 with sa and sb as scale tiles (quant_mxfp4_1x32_tiled or
    fp4_scales_to_tiles)."""
    M, N, K = _fp4_tiled_operands(aq, sa, bq, sb, 32)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=aq.device)
    _need_cuda("out", out, out_dtype)
    if out.shape != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] with contiguous rows")
    st = _lib.fgq_gemm_mxfp4_tiled(aq.data_ptr(), sa.data_ptr(), bq.data_ptr(), sb.data_ptr(),
                                   out.data_ptr(), out.stride(0), M, N, K,
                                   FGQ_OUT_BF16 if out_dtype == torch.bfloat16 else FGQ_OUT_F32,
                                   _stream(aq))
    check("fgq_gemm_mxfp4_tiled", st)
    return out


def gemm_nvfp4_tiled(aq: torch.Tensor, sa: torch.Tensor, ga: torch.Tensor, bq: torch.Tensor,
                     sb: torch.Tensor, gb: torch.Tensor, out_dtype=torch.float32,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """gemm_nvfp4 with sa and sb as scale tiles (quant_nvfp4_1x16_tiled or
    fp4_scales_to_tiles)."""
    M, N, K = _fp4_tiled_operands(aq, sa, bq, sb, 16)
    _need_cuda("ga", ga, torch.float32)
    _need_cuda("gb", gb, torch.float32)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=aq.device)
    _need_cuda("out", out, out_dtype)
    if out.shape != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] with contiguous rows")
    st = _lib.fgq_gemm_nvfp4_tiled(aq.data_ptr(), sa.data_ptr(), ga.data_ptr(), bq.data_ptr(),
                                   sb.data_ptr(), gb.data_ptr(), out.data_ptr(), out.stride(0), M,
                                   N, K, FGQ_OUT_BF16 if out_dtype == torch.bfloat16 else FGQ_OUT_F32,
                                   _stream(aq))
    check("fgq_gemm_nvfp4_tiled", st)
    return out


def ue8m0_scale_tiles_bytes(R: int, K: int) -> int:
    """Bytes of UE8M0 code tiles for R rows and reduction length K."""
    st, n = _lib.fgq_ue8m0_scale_tiles_bytes(R, K)
    check("fgq_ue8m0_scale_tiles_bytes", st)
    return n


def ue8m0_scale_tiles(s: torch.Tensor, weight: bool, tiles: torch.Tensor | None = None):
    """UE8M0 code tiles from fp32 power-of-two scales: activation scales
    s [M, K/128] (weight=False) or weight scales s [K/128, N/128]
    (weight=True, one row of codes per column of the weight).  Returns a
    1-D uint8 tensor for gemm_fp8_ue8m0_tiled."""
    _need_cuda("s", s, torch.float32)
    if s.dim() != 2 or not s.is_contiguous():
        raise ValueError("s must be a dense 2-D tensor")
    if weight:
        K, N = 128 * s.shape[0], 128 * s.shape[1]
        R = N
    else:
        R, K = s.shape[0], 128 * s.shape[1]
    n = ue8m0_scale_tiles_bytes(R, K)
    tiles = _tiles_out(tiles, n, s.device, "tiles")
    if weight:
        st = _lib.fgq_ue8m0_scale_tiles_weight(s.data_ptr(), K, N, tiles.data_ptr(), _stream(s))
    else:
        st = _lib.fgq_ue8m0_scale_tiles_act(s.data_ptr(), R, K, tiles.data_ptr(), _stream(s))
    check("fgq_ue8m0_scale_tiles", st)
    return tiles


def quant_operands_ue8m0_tiles(x: torch.Tensor, w: torch.Tensor, xq: torch.Tensor | None = None,
                               sa_tiles: torch.Tensor | None = None,
                               wq: torch.Tensor | None = None,
                               sb_tiles: torch.Tensor | None = None):
    """quant_operands(x, w, "ue8m0") with the scales written as the UE8M0
    code tiles gemm_fp8_ue8m0_tiled takes.  Returns (xq, sa_tiles, wq,
    sb_tiles)."""
    _need_cuda("x", x, torch.bfloat16)
    _need_cuda("w", w, torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1 or w.dim() != 2 or w.stride(1) != 1:
        raise ValueError("x and w must be 2-D with a contiguous last dimension")
    M, K = x.shape
    K2, N = w.shape
    if K2 != K:
        raise ValueError(f"x is [M, {K}] but w is [{K2}, N]")
    dev = x.device
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev) if xq is None else xq
    wq = torch.empty((N, K), dtype=torch.uint8, device=dev) if wq is None else wq
    _need_cuda("xq", xq, torch.uint8)
    _need_cuda("wq", wq, torch.uint8)
    if xq.shape != (M, K) or xq.stride(1) != 1 or wq.shape != (N, K) or not wq.is_contiguous():
        raise ValueError("xq must be [M, K] (contiguous rows) and wq a dense [N, K]")
    sa_tiles = _tiles_out(sa_tiles, ue8m0_scale_tiles_bytes(M, K), dev, "sa_tiles")
    sb_tiles = _tiles_out(sb_tiles, ue8m0_scale_tiles_bytes(N, K), dev, "sb_tiles")
    st = _lib.fgq_quant_operands_ue8m0_tiles(x.data_ptr(), M, K, x.stride(0), xq.data_ptr(),
                                             xq.stride(0), sa_tiles.data_ptr(), w.data_ptr(), N,
                                             w.stride(0), wq.data_ptr(), sb_tiles.data_ptr(),
                                             _stream(x))
    check("fgq_quant_operands_ue8m0_tiles", st)
    return xq, sa_tiles, wq, sb_tiles


def gemm_fp8_ue8m0_tiled(aq: torch.Tensor, sa_tiles: torch.Tensor, bq: torch.Tensor,
                         sb_tiles: torch.Tensor, out_dtype=torch.bfloat16,
                         out: torch.Tensor | None = None) -> torch.Tensor:
    """The power-of-two-scale FP8 GEMM with UE8M0 code tiles: aq [M, K] and
    bq [N, K] E4M3 codes (bq as quant_w_128x128 returns it), sa_tiles and
    sb_tiles from ue8m0_scale_tiles."""
    for name, t in (("aq", aq), ("bq", bq), ("sa_tiles", sa_tiles), ("sb_tiles", sb_tiles)):
        _need_cuda(name, t, torch.uint8)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    M, K = aq.shape
    N = bq.shape[0]
    if bq.shape != (N, K):
        raise ValueError("shape mismatch: aq [M, K], bq [N, K]")
    if sa_tiles.numel() != ue8m0_scale_tiles_bytes(M, K) or \
            sb_tiles.numel() != ue8m0_scale_tiles_bytes(N, K):
        raise ValueError("sa_tiles / sb_tiles must be ue8m0_scale_tiles of A and of the weight")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=aq.device)
    _need_cuda("out", out, out_dtype)
    if out.shape != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] with contiguous rows")
    st = _lib.fgq_gemm_fp8_ue8m0_tiled(aq.data_ptr(), sa_tiles.data_ptr(), bq.data_ptr(),
                                       sb_tiles.data_ptr(), out.data_ptr(), out.stride(0), M, N, K,
                                       FGQ_OUT_BF16 if out_dtype == torch.bfloat16 else FGQ_OUT_F32,
                                       _stream(aq))
    check("fgq_gemm_fp8_ue8m0_tiled", st)
    return out


def splitk_workspace(M: int, N: int, K: int, device=None) -> torch.Tensor:
    """A zero-filled workspace for gemm_fp8_blockscaled_splitk on `device`."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        st, n = _lib.fgq_gemm_splitk_workspace_size(M, N, K)
    check("fgq_gemm_splitk_workspace_size", st)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=dev)


def gemm_fp8_blockscaled_splitk(aq: torch.Tensor, sa: torch.Tensor, bq: torch.Tensor,
                                sb: torch.Tensor, workspace: torch.Tensor, out_dtype=torch.float32,
                                mode="fp32", out: torch.Tensor | None = None) -> torch.Tensor:
    """gemm_fp8_blockscaled with split-K over a caller-owned workspace (see
    splitk_workspace); deterministic, for M <= 256."""
    M, K = aq.shape
    N = bq.shape[0]
    _need_cuda("workspace", workspace, torch.uint8)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=aq.device)
    for name, t in (("aq", aq), ("bq", bq), ("sa", sa), ("sb", sb)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    st = _lib.fgq_gemm_fp8_blockscaled_splitk(
        aq.data_ptr(), sa.data_ptr(), bq.data_ptr(), sb.data_ptr(), out.data_ptr(), out.stride(0),
        M, N, K, FGQ_OUT_BF16 if out.dtype == torch.bfloat16 else FGQ_OUT_F32, scale_mode(mode),
        workspace.data_ptr(), workspace.numel(), _stream(aq))
    check("fgq_gemm_fp8_blockscaled_splitk", st)
    return out


def device_error(clear: bool = True) -> int:
    """The library's device error word (0 = no kernel gave up on a wait)."""
    st, word = _lib.fgq_device_error(clear)
    if st not in (_lib.FGQ_OK, _lib.FGQ_ERR_DEVICE_TIMEOUT):
        raise FgqError("fgq_device_error", st)
    return word
