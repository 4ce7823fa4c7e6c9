"""Narrow floating-point formats, written out from their definitions.

All rounding here is IEEE 754 round-to-nearest, ties-to-even, applied ONCE to
an exact float64 input.  A binary format is described by its precision p
(significand bits including the implicit one), its minimum normal exponent
emin and its largest finite value.  A value is rounded by choosing the
exponent of its leading bit (never below emin, which yields the subnormal
grid), scaling so that the format's unit in the last place is 1, rounding to
an integer with numpy's ``rint`` (ties to even) and scaling back.  Every step
except ``rint`` is a multiplication by a power of two, exact in float64.

Formats:
  bf16     p=8,  emin=-126, max=(2-2^-7)*2^127, overflow -> inf
  fp16     p=11, emin=-14,  max=65504,          overflow -> inf
  e4m3     p=4,  emin=-6,   max=448, no infinity; "satfinite" clamps to +-448
           (OCP 8-bit floating point, E4M3 variant used by tensor cores)
  e2m1     p=2,  emin=0,    max=6; clamps to +-6 (OCP Microscaling v1.0, FP4)
  e8m0     value 2^(b-127) for b in [0,254], b=255 is NaN (OCP MX scale type)

The Humming pages name these formats (INT4 vs NVFP4, MXFP4 weights, FP8
activations: kinachrichten.com, "Warum quantisierte Kernel wichtig sind" and
the W4A8-MXFP4 paragraph of "Kompilierzeiten und gerätespezifisches Tuning")
but do not define them; the definitions above are the formats' own.
"""

from __future__ import annotations

import numpy as np

BF16 = dict(p=8, emin=-126, maxval=float.fromhex("0x1.fep127"), sat=False)
FP16 = dict(p=11, emin=-14, maxval=65504.0, sat=False)
E4M3 = dict(p=4, emin=-6, maxval=448.0, sat=True)
E2M1 = dict(p=2, emin=0, maxval=6.0, sat=True)


def round_to(x, p: int, emin: int, maxval: float, sat: bool) -> np.ndarray:
    """Round float64 values to a binary format, RNE, returning float64 values.

    ``sat`` selects clamping to +-maxval instead of overflow to infinity."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    fin = np.isfinite(x) & (x != 0)
    xf = x[fin]
    _, e = np.frexp(np.abs(xf))          # |x| = f * 2^e, f in [0.5, 1)
    lead = np.maximum(e - 1, emin)        # exponent of the leading bit, >= emin
    ulp_exp = lead - (p - 1)
    r = np.ldexp(np.rint(np.ldexp(xf, -ulp_exp)), ulp_exp)
    big = np.abs(r) > maxval
    if sat:
        r = np.where(big, np.copysign(maxval, r), r)
    else:
        r = np.where(big, np.copysign(np.inf, r), r)
    out[fin] = r
    if sat:
        out = np.where(np.isinf(x), np.copysign(maxval, x), out)
    return out


def bf16(x) -> np.ndarray:
    return round_to(x, **BF16)


def fp16(x) -> np.ndarray:
    return round_to(x, **FP16)


def e4m3(x) -> np.ndarray:
    """Round to e4m3 with saturation (the ``satfinite`` conversion)."""
    return round_to(x, **E4M3)


def e2m1(x) -> np.ndarray:
    """Round to e2m1 with saturation at +-6."""
    return round_to(x, **E2M1)


def round_dtype(name: str):
    """Rounding function for an activation/scale dtype name."""
    return {"bf16": bf16, "fp16": fp16}[name]


# ---------------------------------------------------------------- bit codes

def decode_e4m3(code) -> np.ndarray:
    """Value of an e4m3 byte: s eeee mmm, bias 7, subnormals at e=0,
    0x7F / 0xFF are NaN, no infinities."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return s * mag


def decode_e2m1(code) -> np.ndarray:
    """Value of an e2m1 nibble: s ee m, bias 1, subnormal at e=0."""
    c = np.asarray(code, dtype=np.int64) & 0xF
    s = np.where(c >> 3, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m / 2.0, e - 1))
    return s * mag


def decode_e8m0(code) -> np.ndarray:
    """Value of an e8m0 byte: 2^(b-127); 0xFF is NaN."""
    b = np.asarray(code, dtype=np.int64) & 0xFF
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


def _encode_by_table(values, table: np.ndarray, nbits: int) -> np.ndarray:
    """Code of each (already representable) value by exact table lookup.

    In both e4m3 and e2m1 the positive codes 0 .. 2^(nbits-1)-1 are ordered by
    magnitude and the top bit is the sign, so the magnitude is located with a
    binary search over the positive half of the table and must match exactly.
    Zero keeps the sign of the input (-0.0 -> the negative-zero code)."""
    v = np.asarray(values, dtype=np.float64)
    half = 1 << (nbits - 1)
    pos = table[:half]
    finite = ~np.isnan(pos)
    pos = pos[finite]
    mag = np.abs(v)
    idx = np.searchsorted(pos, mag)
    idx = np.minimum(idx, pos.size - 1)
    if np.isnan(v).any() or not np.array_equal(pos[idx], mag):
        raise ValueError(f"values are not representable in the {nbits}-bit format")
    return idx.astype(np.int64) | np.where(np.signbit(v), half, 0)


E4M3_TABLE = decode_e4m3(np.arange(256))
E2M1_TABLE = decode_e2m1(np.arange(16))


def encode_e4m3(x) -> np.ndarray:
    """e4m3 byte of round-to-nearest-even, saturating (satfinite) of x."""
    return _encode_by_table(e4m3(x), E4M3_TABLE, 8).astype(np.uint8)


def encode_e2m1(x) -> np.ndarray:
    """e2m1 nibble of round-to-nearest-even, saturating at +-6, of x."""
    return _encode_by_table(e2m1(x), E2M1_TABLE, 4).astype(np.uint8)


def bf16_bits(x) -> np.ndarray:
    """uint16 bit pattern of bf16 values (x must already be representable)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    if not np.array_equal(f.astype(np.float64), np.asarray(x, dtype=np.float64), equal_nan=True):
        raise ValueError("values are not representable in bf16")
    bits = f.view(np.uint32)
    if np.any(bits & 0xFFFF):
        raise ValueError("values are not representable in bf16")
    return (bits >> 16).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint32) << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def fp16_bits(x) -> np.ndarray:
    """uint16 bit pattern of fp16 values (x must already be representable)."""
    h = np.asarray(x, dtype=np.float64).astype(np.float16)
    if not np.array_equal(h.astype(np.float64), np.asarray(x, dtype=np.float64), equal_nan=True):
        raise ValueError("values are not representable in fp16")
    return h.view(np.uint16)


def fp16_from_bits(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def dtype_bits(name: str, x) -> np.ndarray:
    return {"bf16": bf16_bits, "fp16": fp16_bits}[name](x)


def dtype_from_bits(name: str, bits) -> np.ndarray:
    return {"bf16": bf16_from_bits, "fp16": fp16_from_bits}[name](bits)
