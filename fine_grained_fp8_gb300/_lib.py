"""ctypes binding of libfgq.so (C ABI in include/fgq.h).

Argument marshalling only: every step of the quantizers and the GEMM runs in
the library's CUDA kernels.  There is no fallback of any kind: if the shared
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

FGQ_OK = 0
FGQ_ERR_INVALID_ARG = 1
FGQ_ERR_UNSUPPORTED = 2
FGQ_ERR_CUDA = 3
FGQ_ERR_DEVICE_TIMEOUT = 4

FGQ_SCALE_FP32 = 0
FGQ_SCALE_UE8M0 = 1
FGQ_OUT_F32 = 0
FGQ_OUT_BF16 = 1

# Size of the fixed array behind fgq_gemm_fp8_blockscaled_splitk_noalloc.
FGQ_NOALLOC_SCRATCH_BYTES = 16 << 20

# Every symbol include/fgq.h declares, with (restype, argtypes).
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
SIGNATURES = {
    "fgq_quant_act_1x128": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _int, _vp]),
    "fgq_quant_act_128x1": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _int, _vp]),
    "fgq_quant_mxfp4_1x32": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "fgq_nvfp4_global_scale": (_int, [_vp, _i64, _i64, _i64, _vp, _vp]),
    "fgq_quant_nvfp4_1x16": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "fgq_quant_w_128x128": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _int, _vp]),
    "fgq_quant_operands": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _i64, _i64, _vp,
                                  _vp, _int, _vp]),
    "fgq_gemm_fp8_blockscaled": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "fgq_gemm_fp8_blockscaled_ex": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                           _int, _int, _vp]),
    "fgq_gemm_fp8_blockscaled_splitk": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                               _int, _int, _vp, ctypes.c_size_t, _vp]),
    "fgq_gemm_splitk_workspace_size": (_int, [_i64, _i64, _i64, ctypes.POINTER(ctypes.c_size_t)]),
    "fgq_gemm_mxfp4": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, _vp]),
    "fgq_gemm_nvfp4": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int,
                              _vp]),
    "fgq_gemm_mxfp4_tiled": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, _vp]),
    "fgq_gemm_nvfp4_tiled": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                    _int, _vp]),
    "fgq_quant_mxfp4_1x32_tiled": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "fgq_quant_nvfp4_1x16_tiled": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "fgq_fp4_scale_tiles_bytes": (_int, [_i64, _i64, ctypes.POINTER(ctypes.c_size_t)]),
    "fgq_fp4_scales_to_tiles": (_int, [_vp, _i64, _i64, _vp, _vp]),
    "fgq_ue8m0_scale_tiles_bytes": (_int, [_i64, _i64, ctypes.POINTER(ctypes.c_size_t)]),
    "fgq_ue8m0_scale_tiles_act": (_int, [_vp, _i64, _i64, _vp, _vp]),
    "fgq_quant_operands_ue8m0_tiles": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _i64,
                                              _i64, _vp, _vp, _vp]),
    "fgq_ue8m0_scale_tiles_weight": (_int, [_vp, _i64, _i64, _vp, _vp]),
    "fgq_gemm_fp8_ue8m0_tiled": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int,
                                        _vp]),
    "fgq_gemm_fp8_blockscaled_fused_act": (_int, [_vp, _i64, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                                  _int, _int, _vp]),
    "fgq_gemm_fp8_blockscaled_splitk_noalloc": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                                       _i64, _int, _int, _vp]),
    "fgq_selftest_wait_timeout": (_int, [_vp]),
    "fgq_status_string": (ctypes.c_char_p, [_int]),
    "fgq_device_error": (_int, [ctypes.POINTER(ctypes.c_uint32), _int]),
    "fgq_version": (_int, []),
}

_lock = threading.Lock()
_lib = None


class FgqError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: status {status} ({status_string(status)})")


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libfgq.so (built by fine_grained_fp8_gb300.build.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libfgq.so not found at {p}: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().fgq_status_string(int(status)).decode()
    except Exception:  # library not loadable: still give the code
        return "unknown"


def check(func: str, status: int) -> None:
    if status != FGQ_OK:
        raise FgqError(func, status)


# Raw C-ABI calls under their C names (pointers as ints, stream as int handle).

def fgq_quant_act_1x128(x, M, K, ldx, xq, ldq, sx, mode, stream) -> int:
    return load().fgq_quant_act_1x128(x, M, K, ldx, xq, ldq, sx, mode, stream)


def fgq_quant_act_128x1(x, M, K, ldx, xqt, sxt, mode, stream) -> int:
    return load().fgq_quant_act_128x1(x, M, K, ldx, xqt, sxt, mode, stream)


def fgq_quant_mxfp4_1x32(x, R, K, ldx, xq, sx, stream) -> int:
    return load().fgq_quant_mxfp4_1x32(x, R, K, ldx, xq, sx, stream)


def fgq_nvfp4_global_scale(x, R, K, ldx, g, stream) -> int:
    return load().fgq_nvfp4_global_scale(x, R, K, ldx, g, stream)


def fgq_quant_nvfp4_1x16(x, R, K, ldx, g, xq, sx, stream) -> int:
    return load().fgq_quant_nvfp4_1x16(x, R, K, ldx, g, xq, sx, stream)


def fgq_quant_w_128x128(w, K, N, ldw, wq, sw, mode, stream) -> int:
    return load().fgq_quant_w_128x128(w, K, N, ldw, wq, sw, mode, stream)


def fgq_quant_operands(x, M, K, ldx, xq, ldq, sx, w, N, ldw, wq, sw, mode, stream) -> int:
    return load().fgq_quant_operands(x, M, K, ldx, xq, ldq, sx, w, N, ldw, wq, sw, mode, stream)


def fgq_gemm_fp8_blockscaled(A, sA, B, sB, C, M, N, K, stream) -> int:
    return load().fgq_gemm_fp8_blockscaled(A, sA, B, sB, C, M, N, K, stream)


def fgq_gemm_fp8_blockscaled_ex(A, sA, B, sB, C, ldc, M, N, K, out, mode, stream) -> int:
    return load().fgq_gemm_fp8_blockscaled_ex(A, sA, B, sB, C, ldc, M, N, K, out, mode, stream)


def fgq_gemm_fp8_blockscaled_splitk(A, sA, B, sB, C, ldc, M, N, K, out, mode, workspace,
                                    workspace_bytes, stream) -> int:
    return load().fgq_gemm_fp8_blockscaled_splitk(A, sA, B, sB, C, ldc, M, N, K, out, mode,
                                                  workspace, workspace_bytes, stream)


def fgq_gemm_fp8_blockscaled_splitk_noalloc(A, sA, B, sB, C, ldc, M, N, K, out, mode,
                                            stream) -> int:
    return load().fgq_gemm_fp8_blockscaled_splitk_noalloc(A, sA, B, sB, C, ldc, M, N, K, out,
                                                          mode, stream)


def fgq_gemm_fp8_blockscaled_fused_act(A, lda, B, sB, C, ldc, M, N, K, out, mode, stream) -> int:
    return load().fgq_gemm_fp8_blockscaled_fused_act(A, lda, B, sB, C, ldc, M, N, K, out, mode,
                                                     stream)


def fgq_gemm_mxfp4(A, sA, B, sB, C, ldc, M, N, K, out, stream) -> int:
    return load().fgq_gemm_mxfp4(A, sA, B, sB, C, ldc, M, N, K, out, stream)


def fgq_gemm_nvfp4(A, sA, gA, B, sB, gB, C, ldc, M, N, K, out, stream) -> int:
    return load().fgq_gemm_nvfp4(A, sA, gA, B, sB, gB, C, ldc, M, N, K, out, stream)


def fgq_gemm_mxfp4_tiled(A, sA, B, sB, C, ldc, M, N, K, out, stream) -> int:
    return load().fgq_gemm_mxfp4_tiled(A, sA, B, sB, C, ldc, M, N, K, out, stream)


def fgq_gemm_nvfp4_tiled(A, sA, gA, B, sB, gB, C, ldc, M, N, K, out, stream) -> int:
    return load().fgq_gemm_nvfp4_tiled(A, sA, gA, B, sB, gB, C, ldc, M, N, K, out, stream)


def fgq_quant_mxfp4_1x32_tiled(x, R, K, ldx, xq, s_tiles, stream) -> int:
    return load().fgq_quant_mxfp4_1x32_tiled(x, R, K, ldx, xq, s_tiles, stream)


def fgq_quant_nvfp4_1x16_tiled(x, R, K, ldx, g, xq, s_tiles, stream) -> int:
    return load().fgq_quant_nvfp4_1x16_tiled(x, R, K, ldx, g, xq, s_tiles, stream)


def fgq_fp4_scale_tiles_bytes(R, F):
    n = ctypes.c_size_t(0)
    st = load().fgq_fp4_scale_tiles_bytes(R, F, ctypes.byref(n))
    return st, int(n.value)


def fgq_fp4_scales_to_tiles(s, R, F, tiles, stream) -> int:
    return load().fgq_fp4_scales_to_tiles(s, R, F, tiles, stream)


def fgq_ue8m0_scale_tiles_bytes(R, K):
    n = ctypes.c_size_t(0)
    st = load().fgq_ue8m0_scale_tiles_bytes(R, K, ctypes.byref(n))
    return st, int(n.value)


def fgq_quant_operands_ue8m0_tiles(x, M, K, ldx, xq, ldq, sA_tiles, w, N, ldw, wq, sB_tiles,
                                   stream) -> int:
    return load().fgq_quant_operands_ue8m0_tiles(x, M, K, ldx, xq, ldq, sA_tiles, w, N, ldw, wq,
                                                 sB_tiles, stream)


def fgq_ue8m0_scale_tiles_act(sA, M, K, tiles, stream) -> int:
    return load().fgq_ue8m0_scale_tiles_act(sA, M, K, tiles, stream)


def fgq_ue8m0_scale_tiles_weight(sB, K, N, tiles, stream) -> int:
    return load().fgq_ue8m0_scale_tiles_weight(sB, K, N, tiles, stream)


def fgq_gemm_fp8_ue8m0_tiled(A, sA, B, sB, C, ldc, M, N, K, out, stream) -> int:
    return load().fgq_gemm_fp8_ue8m0_tiled(A, sA, B, sB, C, ldc, M, N, K, out, stream)


def fgq_gemm_splitk_workspace_size(M, N, K):
    n = ctypes.c_size_t(0)
    st = load().fgq_gemm_splitk_workspace_size(M, N, K, ctypes.byref(n))
    return st, int(n.value)


def fgq_device_error(clear: bool = True):
    word = ctypes.c_uint32(0)
    st = load().fgq_device_error(ctypes.byref(word), 1 if clear else 0)
    return st, int(word.value)


def fgq_selftest_wait_timeout(stream) -> int:
    return load().fgq_selftest_wait_timeout(stream)


def fgq_version() -> int:
    return load().fgq_version()
