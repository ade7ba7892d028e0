"""CPU oracle for fine-grained FP8 quantization and the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference arm are the only callers.  The
library (``fine_grained_fp8_gb300``) never imports this package, and this
package never imports the library: the two share no code.  The arithmetic
lives in ``fgq_oracle.c`` (plain C, compiled with gcc on first use); this
module only marshals numpy arrays into it.

What each function follows ("Fine-Grained FP8/FP4 Quantization" page):
  quant_act_1x128   §Scaling Granularities (per-tile 1x128) and
                    §DeepGEMM (scale_A[M, K/128])
  quant_w_128x128   §Scaling Granularities (per-block 128x128) and
                    §DeepGEMM (scale_B[K/128, N/128])
  e4m3_*            §UE8M0 vs E4M3 Scale Formats (E4M3 range ~0..448)
  ue8m0_*           §Blackwell: Native Block Scaling (2^(e-127), 4 per word)
  gemm_*            §DeepGEMM: C += partial * scale_A * scale_B per
                    128-wide K chunk, i.e. the fp64 dequantised product.
  fp4_scale_tiles   the FP4 block scales in the library's tiled storage
                    layout (a permutation; its definition is in the
                    docstring).

Parity is pinned for every function (tests/test_oracle_pins.py); nothing
here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MODE_FP32 = 0
MODE_UE8M0 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fgq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile fgq_oracle.c into oracle/_build/liboracle.so with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"],
            check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.fgqo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.fgqo_e4m3_decode.restype = ctypes.c_double
        lib.fgqo_e4m3_encode.argtypes = [ctypes.c_float]
        lib.fgqo_e4m3_encode.restype = ctypes.c_uint8
        lib.fgqo_pow2_ceil.argtypes = [ctypes.c_float]
        lib.fgqo_pow2_ceil.restype = ctypes.c_float
        lib.fgqo_scale_from_amax.argtypes = [ctypes.c_float, ctypes.c_int]
        lib.fgqo_scale_from_amax.restype = ctypes.c_float
        lib.fgqo_ue8m0_code.argtypes = [ctypes.c_float]
        lib.fgqo_ue8m0_code.restype = ctypes.c_int
        lib.fgqo_ue8m0_pack4.argtypes = [_u8p]
        lib.fgqo_ue8m0_pack4.restype = ctypes.c_uint32
        lib.fgqo_ue8m0_unpack.argtypes = [ctypes.c_uint32, ctypes.c_int]
        lib.fgqo_ue8m0_unpack.restype = ctypes.c_double
        lib.fgqo_bf16_to_float.argtypes = [ctypes.c_uint16]
        lib.fgqo_bf16_to_float.restype = ctypes.c_float
        lib.fgqo_quant_act_1x128.argtypes = [_u16p, _i64, _i64, _u8p, _f32p, ctypes.c_int]
        lib.fgqo_quant_act_1x128.restype = ctypes.c_int
        lib.fgqo_quant_act_128x1.argtypes = [_u16p, _i64, _i64, _u8p, _f32p, ctypes.c_int]
        lib.fgqo_quant_act_128x1.restype = ctypes.c_int
        lib.fgqo_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.fgqo_e2m1_decode.restype = ctypes.c_double
        lib.fgqo_e2m1_encode.argtypes = [ctypes.c_double]
        lib.fgqo_e2m1_encode.restype = ctypes.c_uint8
        lib.fgqo_quant_mxfp4_1x32.argtypes = [_u16p, _i64, _i64, _u8p, _u8p]
        lib.fgqo_quant_mxfp4_1x32.restype = ctypes.c_int
        lib.fgqo_gemm_mxfp4.argtypes = [_u8p, _u8p, _u8p, _u8p, _i64, _i64, _i64,
                                        ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_double)]
        lib.fgqo_gemm_mxfp4.restype = ctypes.c_int
        lib.fgqo_gemm_mxfp4_at.argtypes = [_u8p, _u8p, _u8p, _u8p, _i64, _i64, _i64,
                                           ctypes.POINTER(ctypes.c_int64),
                                           ctypes.POINTER(ctypes.c_int64), _i64,
                                           ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_double)]
        lib.fgqo_gemm_mxfp4_at.restype = ctypes.c_int
        lib.fgqo_nvfp4_global_scale.argtypes = [_u16p, _i64, _i64]
        lib.fgqo_nvfp4_global_scale.restype = ctypes.c_float
        lib.fgqo_quant_nvfp4_1x16.argtypes = [_u16p, _i64, _i64, ctypes.c_float, _u8p, _u8p]
        lib.fgqo_quant_nvfp4_1x16.restype = ctypes.c_int
        lib.fgqo_gemm_nvfp4.argtypes = [_u8p, _u8p, ctypes.c_float, _u8p, _u8p, ctypes.c_float,
                                        _i64, _i64, _i64, _f64p, _f64p]
        lib.fgqo_gemm_nvfp4.restype = ctypes.c_int
        lib.fgqo_gemm_nvfp4_at.argtypes = [_u8p, _u8p, ctypes.c_float, _u8p, _u8p, ctypes.c_float,
                                           _i64, _i64, _i64, _i64p, _i64p, _i64, _f64p, _f64p]
        lib.fgqo_gemm_nvfp4_at.restype = ctypes.c_int
        lib.fgqo_quant_w_128x128.argtypes = [_u16p, _i64, _i64, _u8p, _f32p, ctypes.c_int]
        lib.fgqo_quant_w_128x128.restype = ctypes.c_int
        lib.fgqo_gemm_dequant.argtypes = [_u8p, _f32p, _u8p, _f32p, _i64, _i64, _i64,
                                          _f64p, _f64p]
        lib.fgqo_gemm_dequant.restype = ctypes.c_int
        lib.fgqo_gemm_dequant_at.argtypes = [_u8p, _f32p, _u8p, _f32p, _i64, _i64,
                                             _i64p, _i64p, _i64, _f64p, _f64p]
        lib.fgqo_gemm_dequant_at.restype = None
        lib.fgqo_gemm_chunked.argtypes = [_u8p, _f32p, _u8p, _f32p, _i64, _i64, _i64, _f64p]
        lib.fgqo_gemm_chunked.restype = None
        lib.fgqo_gemm_bruteforce.argtypes = [_u8p, _f32p, _u8p, _f32p, _i64, _i64, _i64,
                                             _f64p]
        lib.fgqo_gemm_bruteforce.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctype)


def _bits16(x) -> np.ndarray:
    """bf16 input as a C-contiguous uint16 bit array (numpy uint16/int16, or a
    torch bfloat16 CPU tensor)."""
    if hasattr(x, "dtype") and str(getattr(x, "dtype")) == "torch.bfloat16":
        import torch  # local: only needed for torch inputs
        x = x.contiguous().view(torch.int16).numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.int16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError("bf16 input must be given as 16-bit patterns")
    return x


# ---- element formats ------------------------------------------------------

def e4m3_decode(code: int) -> float:
    return _load().fgqo_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(v: float) -> int:
    return int(_load().fgqo_e4m3_encode(float(v)))


def e4m3_decode_array(codes: np.ndarray) -> np.ndarray:
    table = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def bf16_to_float(bits: int) -> float:
    return _load().fgqo_bf16_to_float(int(bits) & 0xFFFF)


def pow2_ceil(t: float) -> float:
    return _load().fgqo_pow2_ceil(float(t))


def scale_from_amax(amax: float, mode: int = MODE_FP32) -> float:
    return _load().fgqo_scale_from_amax(float(amax), int(mode))


def ue8m0_code(s: float) -> int:
    return _load().fgqo_ue8m0_code(float(s))


def ue8m0_pack4(codes) -> int:
    arr = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    assert arr.size == 4
    return int(_load().fgqo_ue8m0_pack4(_ptr(arr, _u8p)))


def ue8m0_unpack(packed: int, i: int) -> float:
    return _load().fgqo_ue8m0_unpack(int(packed) & 0xFFFFFFFF, int(i))


# ---- quantizers ------------------------------------------------------------

def quant_act_1x128(x_bf16, mode: int = MODE_FP32):
    """X bf16 [M, K] -> (Xq uint8 [M, K], sX float32 [M, K/128])."""
    x = _bits16(x_bf16)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty((M, K // 128), dtype=np.float32)
    rc = _load().fgqo_quant_act_1x128(_ptr(x, _u16p), M, K, _ptr(q, _u8p), _ptr(s, _f32p),
                                      int(mode))
    if rc != 0:
        raise ValueError(f"oracle quant_act_1x128 failed ({rc}): "
                         "K must be a multiple of 128 and inputs finite")
    return q, s


def quant_act_128x1(x_bf16, mode: int = MODE_FP32):
    """X bf16 [M, K] -> (XqT uint8 [K, M], sXT float32 [K, M/128]): groups of
    128 consecutive rows of one column, written transposed (the A operand of
    a GEMM that reduces over M)."""
    x = _bits16(x_bf16)
    M, K = x.shape
    q = np.empty((K, M), dtype=np.uint8)
    s = np.empty((K, M // 128), dtype=np.float32)
    rc = _load().fgqo_quant_act_128x1(_ptr(x, _u16p), M, K, _ptr(q, _u8p), _ptr(s, _f32p),
                                      int(mode))
    if rc != 0:
        raise ValueError(f"oracle quant_act_128x1 failed ({rc}): "
                         "M and K must be multiples of 128 and inputs finite")
    return q, s


def e2m1_decode(code: int) -> float:
    return _load().fgqo_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return _load().fgqo_e2m1_encode(float(v))


def quant_mxfp4_1x32(x_bf16):
    """X bf16 [R, K] -> (Xq uint8 [R, K/2] E2M1 pairs, low nibble = even
    element; sX uint8 [R, K/32] UE8M0 codes)."""
    x = _bits16(x_bf16)
    R, K = x.shape
    q = np.empty((R, K // 2), dtype=np.uint8)
    s = np.empty((R, K // 32), dtype=np.uint8)
    rc = _load().fgqo_quant_mxfp4_1x32(_ptr(x, _u16p), R, K, _ptr(q, _u8p), _ptr(s, _u8p))
    if rc != 0:
        raise ValueError(f"oracle quant_mxfp4_1x32 failed ({rc}): "
                         "K must be a multiple of 32 and inputs finite")
    return q, s


def gemm_mxfp4(aq, sa, bq, sb):
    """fp64 reference of the MXFP4 GEMM: A [M, K] and B^T [N, K] as quantized
    by quant_mxfp4_1x32 -> (C [M, N], T [M, N])."""
    aq, sa, bq, sb = (np.ascontiguousarray(v, dtype=np.uint8) for v in (aq, sa, bq, sb))
    M, N, K = aq.shape[0], bq.shape[0], 2 * aq.shape[1]
    c = np.empty((M, N), dtype=np.float64)
    t = np.empty((M, N), dtype=np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    rc = _load().fgqo_gemm_mxfp4(_ptr(aq, _u8p), _ptr(sa, _u8p), _ptr(bq, _u8p), _ptr(sb, _u8p),
                                 M, N, K, c.ctypes.data_as(dp), t.ctypes.data_as(dp))
    if rc != 0:
        raise ValueError(f"oracle gemm_mxfp4 failed ({rc})")
    return c, t


def gemm_mxfp4_at(aq, sa, bq, sb, rows, cols):
    """The MXFP4 reference at outputs (rows[i], cols[i]) -> (C [n], T [n])."""
    aq, sa, bq, sb = (np.ascontiguousarray(v, dtype=np.uint8) for v in (aq, sa, bq, sb))
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    M, N, K = aq.shape[0], bq.shape[0], 2 * aq.shape[1]
    c = np.empty(rows.size, dtype=np.float64)
    t = np.empty(rows.size, dtype=np.float64)
    dp, ip = ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)
    rc = _load().fgqo_gemm_mxfp4_at(_ptr(aq, _u8p), _ptr(sa, _u8p), _ptr(bq, _u8p), _ptr(sb, _u8p),
                                    M, N, K, rows.ctypes.data_as(ip), cols.ctypes.data_as(ip),
                                    rows.size, c.ctypes.data_as(dp), t.ctypes.data_as(dp))
    if rc != 0:
        raise ValueError(f"oracle gemm_mxfp4_at failed ({rc})")
    return c, t


def nvfp4_global_scale(x_bf16) -> np.float32:
    """NVFP4 per-tensor scale of X bf16: fl32(amax / 2688), 1 for all zeros."""
    x = _bits16(x_bf16)
    R, K = x.shape
    g = _load().fgqo_nvfp4_global_scale(_ptr(x, _u16p), R, K)
    if not np.isfinite(g):
        raise ValueError("oracle nvfp4_global_scale: inputs must be finite")
    return np.float32(g)


def quant_nvfp4_1x16(x_bf16, g=None):
    """X bf16 [R, K] -> (Xq uint8 [R, K/2] E2M1 pairs, low nibble = even
    element; sX uint8 [R, K/16] E4M3 block-scale codes; g float32 global
    scale).  g defaults to nvfp4_global_scale(X)."""
    x = _bits16(x_bf16)
    R, K = x.shape
    if g is None:
        g = nvfp4_global_scale(x)
    g = np.float32(g)
    q = np.empty((R, K // 2), dtype=np.uint8)
    s = np.empty((R, K // 16), dtype=np.uint8)
    rc = _load().fgqo_quant_nvfp4_1x16(_ptr(x, _u16p), R, K, float(g), _ptr(q, _u8p), _ptr(s, _u8p))
    if rc != 0:
        raise ValueError(f"oracle quant_nvfp4_1x16 failed ({rc}): "
                         "K must be a multiple of 16, g positive and inputs finite")
    return q, s, g


def gemm_nvfp4(aq, sa, ga, bq, sb, gb):
    """fp64 reference of the NVFP4 GEMM: A [M, K] and B^T [N, K] as quantized
    by quant_nvfp4_1x16 (global scales ga, gb) -> (C [M, N], T [M, N])."""
    aq, sa, bq, sb = (np.ascontiguousarray(v, dtype=np.uint8) for v in (aq, sa, bq, sb))
    M, N, K = aq.shape[0], bq.shape[0], 2 * aq.shape[1]
    c = np.empty((M, N), dtype=np.float64)
    t = np.empty((M, N), dtype=np.float64)
    rc = _load().fgqo_gemm_nvfp4(_ptr(aq, _u8p), _ptr(sa, _u8p), float(ga), _ptr(bq, _u8p),
                                 _ptr(sb, _u8p), float(gb), M, N, K, _ptr(c, _f64p), _ptr(t, _f64p))
    if rc != 0:
        raise ValueError(f"oracle gemm_nvfp4 failed ({rc})")
    return c, t


def gemm_nvfp4_at(aq, sa, ga, bq, sb, gb, rows, cols):
    """The NVFP4 reference at outputs (rows[i], cols[i]) -> (C [n], T [n])."""
    aq, sa, bq, sb = (np.ascontiguousarray(v, dtype=np.uint8) for v in (aq, sa, bq, sb))
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    M, N, K = aq.shape[0], bq.shape[0], 2 * aq.shape[1]
    c = np.empty(rows.size, dtype=np.float64)
    t = np.empty(rows.size, dtype=np.float64)
    rc = _load().fgqo_gemm_nvfp4_at(_ptr(aq, _u8p), _ptr(sa, _u8p), float(ga), _ptr(bq, _u8p),
                                    _ptr(sb, _u8p), float(gb), M, N, K, _ptr(rows, _i64p),
                                    _ptr(cols, _i64p), rows.size, _ptr(c, _f64p), _ptr(t, _f64p))
    if rc != 0:
        raise ValueError(f"oracle gemm_nvfp4_at failed ({rc})")
    return c, t


def fp4_scale_tiles(s):
    """FP4 block-scale codes s uint8 [R, F] (F % 4 == 0: MXFP4 F = K/32,
    NVFP4 F = K/16) in the tiled layout the FP4 GEMM's tensor-map loads
    take.  The layout is this library's storage format, not the page's: it
    follows from how the block-scaled MMA reads its factors (row m of a
    128-row tile at TMEM lane m, column m / 32; four factor bytes per
    32-bit cell, §Blackwell: Native Block Scaling) and from the copy that
    puts a 32-row x 16-byte shared-memory tile into all four lane quarters.

    Every code s[r, f] goes to byte
        ((r // 128) * (F // 4) + f // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + f % 4
    of a uint8 array of ceil(R / 128) * 128 * F bytes; the bytes of rows
    R .. (multiple of 128) - 1 are zero here.  A pure permutation: no
    arithmetic on the codes."""
    s = np.ascontiguousarray(s, dtype=np.uint8)
    R, F = s.shape
    if F % 4 != 0:
        raise ValueError("fp4_scale_tiles: F must be a multiple of 4")
    out = np.zeros(((R + 127) // 128) * 128 * F, dtype=np.uint8)
    r = np.arange(R, dtype=np.int64)[:, None]
    f = np.arange(F, dtype=np.int64)[None, :]
    off = ((r // 128) * (F // 4) + f // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + f % 4
    out[off] = s
    return out


def quant_w_128x128(w_bf16, mode: int = MODE_FP32):
    """W bf16 [K, N] -> (Wq uint8 [K, N] logical layout, sW float32 [K/128, N/128])."""
    w = _bits16(w_bf16)
    K, N = w.shape
    q = np.empty((K, N), dtype=np.uint8)
    s = np.empty((K // 128, N // 128), dtype=np.float32)
    rc = _load().fgqo_quant_w_128x128(_ptr(w, _u16p), K, N, _ptr(q, _u8p), _ptr(s, _f32p),
                                      int(mode))
    if rc != 0:
        raise ValueError(f"oracle quant_w_128x128 failed ({rc}): "
                         "K, N must be multiples of 128 and inputs finite")
    return q, s


# ---- GEMM ------------------------------------------------------------------

def _gemm_args(aq, sa, bq, sb):
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    bq = np.ascontiguousarray(bq, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    M, K = aq.shape
    K2, N = bq.shape
    assert K == K2 and K % 128 == 0 and N % 128 == 0
    assert sa.shape == (M, K // 128) and sb.shape == (K // 128, N // 128)
    return aq, sa, bq, sb, M, N, K


def gemm_dequant(aq, sa, bq, sb):
    """fp64 C = A_hat @ B_hat and T = |A_hat| @ |B_hat| (Bq in logical [K, N])."""
    aq, sa, bq, sb, M, N, K = _gemm_args(aq, sa, bq, sb)
    c = np.empty((M, N), dtype=np.float64)
    t = np.empty((M, N), dtype=np.float64)
    rc = _load().fgqo_gemm_dequant(_ptr(aq, _u8p), _ptr(sa, _f32p), _ptr(bq, _u8p),
                                   _ptr(sb, _f32p), M, N, K, _ptr(c, _f64p), _ptr(t, _f64p))
    if rc != 0:
        raise MemoryError("oracle gemm_dequant could not allocate its B_hat buffer")
    return c, t


def gemm_dequant_at(aq, sa, bq, sb, rows, cols):
    """C and T at the listed (rows[i], cols[i]) output positions only."""
    aq, sa, bq, sb, M, N, K = _gemm_args(aq, sa, bq, sb)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    assert rows.shape == cols.shape and rows.ndim == 1
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < M
                              and cols.min() >= 0 and cols.max() < N)
    c = np.empty(rows.size, dtype=np.float64)
    t = np.empty(rows.size, dtype=np.float64)
    _load().fgqo_gemm_dequant_at(_ptr(aq, _u8p), _ptr(sa, _f32p), _ptr(bq, _u8p),
                                 _ptr(sb, _f32p), N, K, _ptr(rows, _i64p), _ptr(cols, _i64p),
                                 rows.size, _ptr(c, _f64p), _ptr(t, _f64p))
    return c, t


def gemm_chunked(aq, sa, bq, sb):
    """The page's per-128-K-chunk form, in fp64 (cross-check of the regrouping)."""
    aq, sa, bq, sb, M, N, K = _gemm_args(aq, sa, bq, sb)
    c = np.empty((M, N), dtype=np.float64)
    _load().fgqo_gemm_chunked(_ptr(aq, _u8p), _ptr(sa, _f32p), _ptr(bq, _u8p),
                              _ptr(sb, _f32p), M, N, K, _ptr(c, _f64p))
    return c


def gemm_bruteforce(aq, sa, bq, sb):
    """Triple loop recomputing every dequantised value (tiny inputs only)."""
    aq, sa, bq, sb, M, N, K = _gemm_args(aq, sa, bq, sb)
    c = np.empty((M, N), dtype=np.float64)
    _load().fgqo_gemm_bruteforce(_ptr(aq, _u8p), _ptr(sa, _f32p), _ptr(bq, _u8p),
                                 _ptr(sb, _f32p), M, N, K, _ptr(c, _f64p))
    return c


def gemm_within_tolerance(c_gpu, c_ref, t_ref, rel: float = 2e-3, out_bf16: bool = False):
    """Elementwise |C - C_ref| <= rel * T; returns (ok, max |err| / bound * rel).

    The bound applies to the fp32 accumulator.  A bf16 output is that
    accumulator rounded to nearest even, which adds at most half a bf16 ulp,
    i.e. 2^-8 of its magnitude (|acc| <= |C_ref| + rel * T), so for bf16
    outputs the bound is rel * T + 2^-8 * (|C_ref| + rel * T)."""
    c_gpu = np.asarray(c_gpu, dtype=np.float64)
    err = np.abs(c_gpu - c_ref)
    bound = rel * t_ref
    if out_bf16:
        bound = bound + 2.0 ** -8 * (np.abs(c_ref) + rel * t_ref)
    ok = bool(np.all(err <= bound)) and bool(np.all(np.isfinite(c_gpu)))
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                         np.where(err > 0, np.inf, 0.0)) * rel
    return ok, float(ratio.max()) if ratio.size else 0.0
