"""The C ABI library loads and exports every symbol include/fgq.h declares;
argument checks reject bad calls before touching any device (no GPU needed)."""
import ctypes
import os
import re

import pytest

from fine_grained_fp8_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "fgq.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fgq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    syms = _declared_symbols()
    for name in ("fgq_quant_act_1x128", "fgq_quant_w_128x128", "fgq_gemm_fp8_blockscaled"):
        assert name in syms


def test_library_exports_every_declared_symbol(fgq):
    lib = fgq.load()
    raw = ctypes.CDLL(_lib.library_path())
    for name in _declared_symbols():
        assert hasattr(raw, name), name
        assert name in _lib.SIGNATURES, f"binding has no signature for {name}"
    assert set(_lib.SIGNATURES) == set(_declared_symbols())
    assert lib.fgq_version() >= 100


def test_status_strings(fgq):
    for code in range(5):
        s = _lib.status_string(code)
        assert s and s != "unknown status"
    assert _lib.status_string(99) == "unknown status"


# Calls the library must refuse before any CUDA call.  Pointers are fake
# (never dereferenced: validation fails first).
P = 0x10000  # 16-byte aligned fake address


@pytest.mark.parametrize("args", [
    (0, 4, 128, 128, P, 128, P, 0, None),        # null x
    (P, 4, 100, 128, P, 128, P, 0, None),        # K % 128
    (P, 4, 0, 128, P, 128, P, 0, None),          # K == 0
    (P, -1, 128, 128, P, 128, P, 0, None),       # M < 0
    (P, 4, 128, 120, P, 128, P, 0, None),        # ldx < K
    (P, 4, 128, 132, P, 128, P, 0, None),        # ldx % 8
    (P, 4, 128, 128, P, 136, P, 0, None),        # ldq % 16
    (P + 2, 4, 128, 128, P, 128, P, 0, None),    # x misaligned
    (P, 4, 128, 128, P + 8, 128, P, 0, None),    # xq misaligned
    (P, 4, 128, 128, P, 128, P, 7, None),        # bad mode
])
def test_quant_act_rejects(fgq, args):
    assert _lib.fgq_quant_act_1x128(*args) == _lib.FGQ_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (P, 4, 128, 128, P, 128, P, 0, 128, 128, P, P, 0, None),      # null w
    (P, 4, 128, 128, P, 128, P, P, 100, 128, P, P, 0, None),      # N % 128
    (P, 4, 100, 128, P, 128, P, P, 128, 128, P, P, 0, None),      # K % 128
    (P, 4, 128, 128, P, 128, P, P, 128, 120, P, P, 0, None),      # ldw < N
    (P, 4, 128, 128, P, 128, P, P, 128, 128, P + 8, P, 0, None),  # wq misaligned
    (0, 4, 128, 128, P, 128, P, P, 128, 128, P, P, 0, None),      # null x (M > 0)
    (P, 4, 128, 128, P, 136, P, P, 128, 128, P, P, 0, None),      # ldq % 16
    (P + 2, 4, 128, 128, P, 128, P, P, 128, 128, P, P, 0, None),  # x misaligned
    (P, -1, 128, 128, P, 128, P, P, 128, 128, P, P, 0, None),     # M < 0
    (P, 4, 128, 128, P, 128, P, P, 128, 128, P, P, 9, None),      # bad mode
])
def test_quant_operands_rejects(fgq, args):
    assert _lib.fgq_quant_operands(*args) == _lib.FGQ_ERR_INVALID_ARG


def test_quant_act_empty_is_ok(fgq):
    assert _lib.fgq_quant_act_1x128(0, 0, 128, 128, 0, 128, 0, 0, None) == _lib.FGQ_OK


@pytest.mark.parametrize("args", [
    (0, 128, 128, 128, P, P, 0, None),
    (P, 100, 128, 128, P, P, 0, None),
    (P, 128, 100, 128, P, P, 0, None),
    (P, 128, 128, 64, P, P, 0, None),
    (P, 128, 128, 132, P, P, 0, None),
    (P + 4, 128, 128, 128, P, P, 0, None),
    (P, 128, 128, 128, P, P, 2, None),
])
def test_quant_w_rejects(fgq, args):
    assert _lib.fgq_quant_w_128x128(*args) == _lib.FGQ_ERR_INVALID_ARG


GEMM_BAD_ARGS = [
    (0, P, P, P, P, 128, 128, 128, 128, 0, 0, None),      # null A
    (P, P, P, P, P, 128, 128, 128, 100, 0, 0, None),      # K % 128
    (P, P, P, P, P, 128, 128, 100, 128, 0, 0, None),      # N % 128
    (P, P, P, P, P, 120, 128, 128, 128, 0, 0, None),      # ldc < N
    (P, P, P, P, P, 130, 128, 128, 128, 0, 0, None),      # ldc % 4 (fp32)
    (P, P, P, P, P, 132, 128, 128, 128, 1, 0, None),      # ldc % 8 (bf16)
    (P, P, P, P, P + 4, 128, 128, 128, 128, 0, 0, None),  # C misaligned
    (P, P, P + 8, P, P, 128, 128, 128, 128, 0, 0, None),  # B misaligned
    (P, P, P, P, P, 128, 128, 128, 128, 2, 0, None),      # bad out dtype
    (P, P, P, P, P, 128, 128, 128, 128, 0, 3, None),      # bad mode
    (P, P, P, P, P, 128, -1, 128, 128, 0, 0, None),       # M < 0
    (P, 0, P, P, P, 128, 128, 128, 128, 0, 0, None),      # null sA
    (P, P, P, 0, P, 128, 128, 128, 128, 0, 0, None),      # null sB
    (P, P, P, P, 0, 128, 128, 128, 128, 0, 0, None),      # null C
    (P, P + 2, P, P, P, 128, 128, 128, 128, 0, 0, None),  # sA misaligned
]


@pytest.mark.parametrize("args", GEMM_BAD_ARGS)
def test_gemm_rejects(fgq, args):
    assert _lib.fgq_gemm_fp8_blockscaled_ex(*args) == _lib.FGQ_ERR_INVALID_ARG


@pytest.mark.parametrize("args", GEMM_BAD_ARGS)
def test_gemm_noalloc_rejects(fgq, args):
    """The entry point without a workspace runs the same checks, all before
    any device call."""
    assert _lib.fgq_gemm_fp8_blockscaled_splitk_noalloc(*args) == _lib.FGQ_ERR_INVALID_ARG


@pytest.mark.parametrize("args", GEMM_BAD_ARGS)
def test_gemm_splitk_rejects(fgq, args):
    a = args[:-1] + (P, 1 << 20) + args[-1:]
    assert _lib.fgq_gemm_fp8_blockscaled_splitk(*a) == _lib.FGQ_ERR_INVALID_ARG


def test_gemm_plain_signature_rejects(fgq):
    assert _lib.fgq_gemm_fp8_blockscaled(P, P, P, P, P, 128, 128, 100, None) == \
        _lib.FGQ_ERR_INVALID_ARG
    assert _lib.fgq_gemm_fp8_blockscaled(P, P, P, P, P, 0, 128, 128, None) == _lib.FGQ_OK


def test_product_path_has_no_oracle_dependency():
    """The library package never imports the oracle (and vice versa)."""
    pkg = os.path.join(ROOT, "fine_grained_fp8_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, f)) as fh:
                    src = fh.read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "fgq_oracle" not in src, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            with open(os.path.join(ROOT, "oracle", f)) as fh:
                src = fh.read()
            assert not re.search(r"^\s*(import|from)\s+fine_grained_fp8_gb300\b", src, re.M), f
            assert "libfgq" not in src, f


@pytest.mark.parametrize("args", [
    (0, 256, 128, 128, P, P, 0, None),       # null x
    (P, 200, 128, 128, P, P, 0, None),       # M % 128
    (P, 256, 100, 128, P, P, 0, None),       # K % 128
    (P, 256, 128, 120, P, P, 0, None),       # ldx < K
    (P, 256, 128, 128, P + 8, P, 0, None),   # xqt misaligned
    (P, 256, 128, 128, P, P, 5, None),       # bad mode
])
def test_quant_128x1_rejects(fgq, args):
    assert _lib.fgq_quant_act_128x1(*args) == _lib.FGQ_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (0, 4, 64, 64, P, P, None),              # null x
    (P, 4, 48, 64, P, P, None),              # K % 32
    (P, -1, 64, 64, P, P, None),             # R < 0
    (P, 4, 64, 60, P, P, None),              # ldx < K
    (P + 2, 4, 64, 64, P, P, None),          # x misaligned
    (P, 4, 64, 64, P + 2, P, None),          # xq misaligned
])
def test_quant_mxfp4_rejects(fgq, args):
    assert _lib.fgq_quant_mxfp4_1x32(*args) == _lib.FGQ_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (0, 4, 64, 64, P, None),                 # null x
    (P, 4, 40, 64, P, None),                 # K % 16
    (P, 4, 64, 64, 0, None),                 # null g
    (P, 4, 64, 60, P, None),                 # ldx < K
    (P, 4, 64, 64, P + 2, None),             # g misaligned
])
def test_nvfp4_global_scale_rejects(fgq, args):
    assert _lib.fgq_nvfp4_global_scale(*args) == _lib.FGQ_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (0, 4, 64, 64, P, P, P, None),           # null x
    (P, 4, 40, 64, P, P, P, None),           # K % 16
    (P, 4, 64, 64, 0, P, P, None),           # null g
    (P, 4, 64, 64, P, P + 2, P, None),       # xq misaligned
    (P, 4, 64, 68, P, P, P, None),           # ldx % 8
])
def test_quant_nvfp4_rejects(fgq, args):
    assert _lib.fgq_quant_nvfp4_1x16(*args) == _lib.FGQ_ERR_INVALID_ARG


def test_fp4_quantizers_empty_is_ok(fgq):
    assert _lib.fgq_quant_mxfp4_1x32(0, 0, 64, 64, 0, 0, None) == _lib.FGQ_OK
    assert _lib.fgq_quant_nvfp4_1x16(0, 0, 64, 64, 0, 0, 0, None) == _lib.FGQ_OK


@pytest.mark.parametrize("args", [
    (0, P, P, P, P, 256, 128, 256, 256, 0, None),      # null A
    (P, P, P, P, P, 256, 128, 256, 192, 0, None),      # K % 128
    (P, P, P, P, P, 256, 128, 192, 256, 0, None),      # N % 128
    (P, P, P, P, P, 200, 128, 256, 256, 0, None),      # ldc < N
    (P, P, P, P, P, 256, 128, 256, 256, 3, None),      # bad out dtype
    (P + 8, P, P, P, P, 256, 128, 256, 256, 0, None),  # A misaligned
    (P, P + 2, P, P, P, 256, 128, 256, 256, 0, None),  # sA misaligned
])
def test_gemm_mxfp4_rejects(fgq, args):
    assert _lib.fgq_gemm_mxfp4(*args) == _lib.FGQ_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (P, P, 0, P, P, P, P, 256, 128, 256, 256, 0, None),      # null gA
    (P, P, P, P, P, 0, P, 256, 128, 256, 256, 0, None),      # null gB
    (P, P, P, P, P, P, P, 256, 128, 256, 192, 0, None),      # K % 128
    (P, P, P, P, P, P, P, 256, 128, 256, 256, 2, None),      # bad out dtype
    (P, P, P + 2, P, P, P, P, 256, 128, 256, 256, 0, None),  # gA misaligned
    (P, P, P, P, P, P, P + 4, 256, 128, 256, 256, 0, None),  # C misaligned
])
def test_gemm_nvfp4_rejects(fgq, args):
    assert _lib.fgq_gemm_nvfp4(*args) == _lib.FGQ_ERR_INVALID_ARG


def test_fp4_gemms_empty_is_ok(fgq):
    assert _lib.fgq_gemm_mxfp4(0, 0, 0, 0, 0, 256, 0, 256, 256, 0, None) == _lib.FGQ_OK
    assert _lib.fgq_gemm_nvfp4(0, 0, 0, 0, 0, 0, 0, 256, 0, 256, 256, 0, None) == _lib.FGQ_OK


@pytest.mark.parametrize("args", [
    (0, 4, 128, 128, P, P, None),            # null x
    (P, 4, 96, 128, P, P, None),             # K % 128
    (P, 4, 128, 120, P, P, None),            # ldx < K
    (P, 4, 128, 128, P + 2, P, None),        # xq misaligned
    (P, 4, 128, 128, P, 0, None),            # null scale tiles
    (P, 4, 128, 128, P, P + 8, None),        # scale tiles not 16-byte aligned
])
def test_quant_mxfp4_tiled_rejects(fgq, args):
    assert _lib.fgq_quant_mxfp4_1x32_tiled(*args) == _lib.FGQ_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (0, 4, 64, 64, P, P, P, None),           # null x
    (P, 4, 48, 64, P, P, P, None),           # K % 64
    (P, 4, 64, 64, 0, P, P, None),           # null g
    (P, 4, 64, 64, P, P, 0, None),           # null scale tiles
    (P, 4, 64, 64, P, P, P + 4, None),       # scale tiles not 16-byte aligned
])
def test_quant_nvfp4_tiled_rejects(fgq, args):
    assert _lib.fgq_quant_nvfp4_1x16_tiled(*args) == _lib.FGQ_ERR_INVALID_ARG


def test_fp4_scale_tiles_bytes(fgq):
    assert _lib.fgq_fp4_scale_tiles_bytes(130, 8) == (_lib.FGQ_OK, 256 * 8)
    assert _lib.fgq_fp4_scale_tiles_bytes(0, 4) == (_lib.FGQ_OK, 0)
    assert _lib.fgq_fp4_scale_tiles_bytes(4, 6)[0] == _lib.FGQ_ERR_INVALID_ARG
    assert _lib.fgq_fp4_scale_tiles_bytes(-1, 4)[0] == _lib.FGQ_ERR_INVALID_ARG
    assert _lib.fgq_fp4_scales_to_tiles(P, 4, 6, P, None) == _lib.FGQ_ERR_INVALID_ARG
    assert _lib.fgq_fp4_scales_to_tiles(P + 2, 4, 8, P, None) == _lib.FGQ_ERR_INVALID_ARG
    assert _lib.fgq_fp4_scales_to_tiles(0, 0, 8, 0, None) == _lib.FGQ_OK


@pytest.mark.parametrize("args", [
    (0, P, P, P, P, 256, 128, 256, 256, 0, None),      # null A
    (P, P, P, P, P, 256, 128, 256, 192, 0, None),      # K % 128
    (P, P, P, P, P, 256, 128, 192, 256, 0, None),      # N % 128
    (P, P + 4, P, P, P, 256, 128, 256, 256, 0, None),  # sA not 16-byte aligned
    (P, P, P, P + 8, P, 256, 128, 256, 256, 0, None),  # sB not 16-byte aligned
])
def test_gemm_mxfp4_tiled_rejects(fgq, args):
    assert _lib.fgq_gemm_mxfp4_tiled(*args) == _lib.FGQ_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (P, P, 0, P, P, P, P, 256, 128, 256, 256, 0, None),      # null gA
    (P, P + 4, P, P, P, P, P, 256, 128, 256, 256, 0, None),  # sA not 16-byte aligned
    (P, P, P, P, P, P, P, 256, 128, 256, 192, 0, None),      # K % 128
])
def test_gemm_nvfp4_tiled_rejects(fgq, args):
    assert _lib.fgq_gemm_nvfp4_tiled(*args) == _lib.FGQ_ERR_INVALID_ARG


def test_fp4_tiled_empty_is_ok(fgq):
    assert _lib.fgq_gemm_mxfp4_tiled(0, 0, 0, 0, 0, 256, 0, 256, 256, 0, None) == _lib.FGQ_OK
    assert _lib.fgq_gemm_nvfp4_tiled(0, 0, 0, 0, 0, 0, 0, 256, 0, 256, 256, 0, None) == _lib.FGQ_OK
    assert _lib.fgq_quant_mxfp4_1x32_tiled(0, 0, 128, 128, 0, 0, None) == _lib.FGQ_OK
    assert _lib.fgq_quant_nvfp4_1x16_tiled(0, 0, 64, 64, 0, 0, 0, None) == _lib.FGQ_OK


def test_ue8m0_scale_tiles_calls(fgq):
    assert _lib.fgq_ue8m0_scale_tiles_bytes(130, 640) == (_lib.FGQ_OK, 2 * 2 * 512)
    assert _lib.fgq_ue8m0_scale_tiles_bytes(128, 7168) == (_lib.FGQ_OK, 14 * 512)
    assert _lib.fgq_ue8m0_scale_tiles_bytes(4, 100)[0] == _lib.FGQ_ERR_INVALID_ARG
    assert _lib.fgq_ue8m0_scale_tiles_act(P, 4, 100, P, None) == _lib.FGQ_ERR_INVALID_ARG
    assert _lib.fgq_ue8m0_scale_tiles_act(P, 4, 128, P + 4, None) == _lib.FGQ_ERR_INVALID_ARG
    assert _lib.fgq_ue8m0_scale_tiles_act(0, 0, 128, 0, None) == _lib.FGQ_OK
    assert _lib.fgq_ue8m0_scale_tiles_weight(P, 128, 96, P, None) == _lib.FGQ_ERR_INVALID_ARG
    assert _lib.fgq_ue8m0_scale_tiles_weight(0, 128, 128, P, None) == _lib.FGQ_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (0, P, P, P, P, 256, 128, 256, 256, 0, None),      # null A
    (P, P, P, P, P, 256, 128, 256, 192, 0, None),      # K % 128
    (P, P, P, P, P, 256, 128, 192, 256, 0, None),      # N % 128
    (P, P + 4, P, P, P, 256, 128, 256, 256, 0, None),  # sA not 16-byte aligned
    (P, P, P, P, P, 200, 128, 256, 256, 0, None),      # ldc < N
    (P, P, P, P, P, 256, 128, 256, 256, 7, None),      # bad out dtype
])
def test_gemm_fp8_ue8m0_tiled_rejects(fgq, args):
    assert _lib.fgq_gemm_fp8_ue8m0_tiled(*args) == _lib.FGQ_ERR_INVALID_ARG


def test_gemm_fp8_ue8m0_tiled_empty_is_ok(fgq):
    assert _lib.fgq_gemm_fp8_ue8m0_tiled(0, 0, 0, 0, 0, 256, 0, 256, 256, 0, None) == _lib.FGQ_OK
