"""Readers for the hand-written fixtures under tests/golden/."""
import os
import struct

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if line and not line.startswith("#"):
                yield line


def e4m3_codes():
    """[(code, value)] with value a float (nan allowed, -0.0 kept)."""
    out = []
    for line in _lines("e4m3_codes.txt"):
        code, value = line.split()
        out.append((int(code, 16), float(value)))
    return out


def float_to_bf16_bits(v: float) -> int:
    bits = struct.unpack("<I", struct.pack("<f", v))[0]
    if bits & 0xFFFF:
        raise ValueError(f"{v!r} is not exactly representable in bf16")
    if struct.unpack("<f", struct.pack("<I", bits))[0] != v:
        raise ValueError(f"{v!r} is not exactly representable in fp32")
    return bits >> 16


def quant_groups():
    """[(name, mode, bf16_bits list, scale_bits, codes list)]."""
    out = []
    for line in _lines("quant_groups.txt"):
        name, mode, values, scale, codes = [p.strip() for p in line.split("|")]
        bits = []
        for tok in values.split():
            if tok.startswith("b:"):
                bits.append(int(tok[2:], 16))
            else:
                bits.append(float_to_bf16_bits(float(tok)))
        out.append((name, mode, bits, int(scale, 16), [int(c, 16) for c in codes.split()]))
    return out
