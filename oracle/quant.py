"""Quantizers, the standard-format encoding and dequantization.

The Humming pages describe a "standard format" into which every exported
checkpoint is converted, holding weights, scales, zero points and further
tensors uniformly (jetabc.cn post, "Humming 的做法", item 1; kinachrichten.com,
"Wie die Architektur funktioniert"), and a representation that fixes "what
stored values and associated scales mean" (retrivium.ai retrospective "vLLM
Humming: why shared quantization still needs specialized kernels", section
"Representation answers a different question").  They give no formulas and no
byte layout, so the following readings are taken (each also listed in the
design notes):

Weights are a logical matrix W[k, n] (K rows, N columns; C = A @ W).

Symmetric INT4 (group g along K, one scale per (group, column)):
    amax = max |W| over the group
    s    = sdt(amax / 7)          (sdt = scale dtype, round to nearest even;
                                   amax == 0 gives s = 1)
    q    = clip(rint(W / s), -8, 7)   using the stored, rounded s
    w^   = adt(q * s)             one rounding to the activation dtype

Asymmetric UINT4 (min/max):
    lo, hi = min W, max W over the group
    s    = sdt((hi - lo) / 15)    (hi == lo gives s = 1)
    z    = clip(rint(-lo / s), 0, 15)
    q    = clip(rint(W / s) + z, 0, 15)
    w^   = adt((q - z) * s)       one rounding

MXFP4 (one e8m0 exponent per 32 consecutive k of one column; OCP MX v1.0):
    E    = floor(log2(amax)) - 2 (2 = the e2m1 maximum exponent), clamped to
           [-127, 127]; b = E + 127;  amax == 0 gives b = 0 and all codes 0
    c    = e2m1_rne_saturating(W / 2^E)
    w^   = e2m1(c) * 2^E          exact in float64

NVFP4 (the pages name NVFP4 as a format whose number format and scaling
differ from INT4's: kinachrichten.com, "Warum quantisierte Kernel wichtig
sind"; they give no definition, so the common one is read: e2m1 elements, one
e4m3 scale per 16 consecutive k of one column, one fp32 scale per tensor):
    t    = fp32(max |W| / (6 * 448))   (6 = e2m1 max, 448 = e4m3 max;
                                        1 when W is all zero)
    s    = e4m3_rne_satfinite(amax / (6 t))   over the block of 16
    c    = e2m1_rne_saturating(W / (s t))     (all 0 when s == 0)
    w^   = e2m1(c) * s * t        exact in float64; the kernel feeds the
                                  exact product e2m1(c) * s (at most five
                                  significant bits, so exact in bf16 and
                                  fp16) to the tensor core and multiplies
                                  the fp32 sum by t

``rint`` rounds half to even.  The product (q - z) * s is exact in float64
(a 5-bit integer times an 8- or 11-bit significand), so w^ is rounded once.

Other integer widths b (the pages list weight-only formats WNA16 with N
free, kinachrichten.com "Warum quantisierte Kernel wichtig sind", and name
GPTQ INT3 as a format the library serves, jetabc.cn post "怎么使用"; they
define neither, so the INT4 rules above are read with 2^b levels):
    symmetric:  s = sdt(amax / (2^(b-1) - 1)),  q = clip(rint(W/s), -2^(b-1), 2^(b-1) - 1)
    asymmetric: s = sdt((hi - lo) / (2^b - 1)), z = clip(rint(-lo/s), 0, 2^b - 1),
                q = clip(rint(W/s) + z, 0, 2^b - 1)
    w^ = adt((q - z) * s), one rounding (at most 9 x 11 significant bits for
    b = 8, exact in float64).

Standard-format encoding (the tensors the library's pack entry point takes):
    qweight int32 [K/8, N]: word (j, n) holds k = 8j + i in bits [4i, 4i+4),
            least significant nibble first; INT4 as 4-bit two's complement,
            UINT4 raw.
    scales  [K/g, N] row-major (group-major), in the scale dtype.
    qzeros  int32 [K/g, N/8]: nibble i of word (G, j) is the zero of column
            8j + i (the stored zero is the true zero, no "-1" offset).
    INT8 / UINT8 (W8A16): qweight int32 [K/4, N]: word (j, n) holds
            k = 4j + i in bits [8i, 8i+8) (two's complement or raw);
            qzeros int32 [K/g, N/4], column 4j + i in byte i of word (G, j).
    INT3 / UINT3 (GPTQ): 32 consecutive codes of a column fill three int32
            words as one little-endian 96-bit stream: k = 32j + i occupies
            bits [3i, 3i+3) of word(3j) | word(3j+1) << 32 | word(3j+2) << 64,
            so qweight is int32 [3K/32, N]; qzeros int32 [K/g, 3N/32] holds
            32 consecutive columns' zeros the same way.
    MXFP4:  codes uint8 [N, K/2]: byte (n, j) holds k = 2j in the low nibble
            and k = 2j + 1 in the high nibble; e2m1 bits are s|e1 e0|m.
            scales uint8 e8m0 [N, K/32].
    NVFP4:  codes as MXFP4; scales uint8 e4m3 [N, K/16]; the tensor scale
            t is one fp32 per matrix (per expert).
"""

from __future__ import annotations

import numpy as np

from . import codecs


def _grouped(w: np.ndarray, g: int) -> np.ndarray:
    """View W[K, N] as [K/g, g, N] (groups along K)."""
    k, n = w.shape
    if k % g:
        raise ValueError("K must be a multiple of the group size")
    return w.reshape(k // g, g, n)


# ------------------------------------------------------------ quantizers

def quantize_int4_sym(w, g: int, sdt: str):
    """Symmetric INT4 quantization.  Returns (q int64 [K,N] in [-8,7],
    s float64 [K/g, N] representable in ``sdt``)."""
    w = np.asarray(w, dtype=np.float64)
    wg = _grouped(w, g)
    amax = np.max(np.abs(wg), axis=1)
    s = codecs.round_dtype(sdt)(amax / 7.0)
    s = np.where(amax == 0, 1.0, s)
    q = np.clip(np.rint(wg / s[:, None, :]), -8, 7)
    return q.reshape(w.shape).astype(np.int64), s


def quantize_uint4_asym(w, g: int, sdt: str):
    """Asymmetric UINT4 quantization with min/max range.  Returns
    (q int64 [K,N] in [0,15], s float64 [K/g,N], z int64 [K/g,N] in [0,15])."""
    w = np.asarray(w, dtype=np.float64)
    wg = _grouped(w, g)
    lo = np.min(wg, axis=1)
    hi = np.max(wg, axis=1)
    s = codecs.round_dtype(sdt)((hi - lo) / 15.0)
    s = np.where(hi == lo, 1.0, s)
    z = np.clip(np.rint(-lo / s), 0, 15)
    q = np.clip(np.rint(wg / s[:, None, :]) + z[:, None, :], 0, 15)
    return q.reshape(w.shape).astype(np.int64), s, z.astype(np.int64)


def quantize_int_sym(w, g: int, sdt: str, bits: int):
    """Symmetric b-bit integer quantization (b = 3, 4 or 8).  Returns
    (q int64 [K,N] in [-2^(b-1), 2^(b-1) - 1], s float64 [K/g, N])."""
    w = np.asarray(w, dtype=np.float64)
    wg = _grouped(w, g)
    top = 2 ** (bits - 1) - 1
    amax = np.max(np.abs(wg), axis=1)
    s = codecs.round_dtype(sdt)(amax / top)
    s = np.where(amax == 0, 1.0, s)
    q = np.clip(np.rint(wg / s[:, None, :]), -top - 1, top)
    return q.reshape(w.shape).astype(np.int64), s


def quantize_uint_asym(w, g: int, sdt: str, bits: int):
    """Asymmetric b-bit quantization with min/max range (b = 3, 4 or 8).
    Returns (q int64 [K,N] in [0, 2^b - 1], s float64 [K/g,N], z int64
    [K/g,N] in [0, 2^b - 1])."""
    w = np.asarray(w, dtype=np.float64)
    wg = _grouped(w, g)
    top = 2 ** bits - 1
    lo = np.min(wg, axis=1)
    hi = np.max(wg, axis=1)
    s = codecs.round_dtype(sdt)((hi - lo) / top)
    s = np.where(hi == lo, 1.0, s)
    z = np.clip(np.rint(-lo / s), 0, top)
    q = np.clip(np.rint(wg / s[:, None, :]) + z[:, None, :], 0, top)
    return q.reshape(w.shape).astype(np.int64), s, z.astype(np.int64)


def quantize_mxfp4(w):
    """MXFP4 quantization along K in blocks of 32.  Returns
    (codes uint8 [K, N] e2m1 nibbles, b uint8 [K/32, N] e8m0 exponents)."""
    w = np.asarray(w, dtype=np.float64)
    wg = _grouped(w, 32)
    amax = np.max(np.abs(wg), axis=1)
    _, e = np.frexp(np.where(amax == 0, 1.0, amax))
    big_e = np.clip(e - 1 - 2, -127, 127)        # floor(log2 amax) - emax(e2m1)
    b = np.where(amax == 0, 0, big_e + 127)
    scale = np.ldexp(1.0, b - 127)
    scaled = wg / scale[:, None, :]                # exact: power-of-two divide
    codes = codecs.encode_e2m1(scaled)
    codes = np.where(amax[:, None, :] == 0, 0, codes)
    return codes.reshape(w.shape).astype(np.uint8), b.astype(np.uint8)


def quantize_nvfp4(w):
    """NVFP4 quantization along K in blocks of 16.  Returns (codes uint8 [K, N]
    e2m1 nibbles, sb uint8 [K/16, N] e4m3 block-scale bytes, t float)."""
    w = np.asarray(w, dtype=np.float64)
    amax_t = float(np.max(np.abs(w))) if w.size else 0.0
    t = float(np.float32(amax_t / (6.0 * 448.0))) if amax_t > 0 else 1.0
    if t == 0.0:                                   # underflow of the fp32 tensor scale
        t = 1.0
    wg = _grouped(w, 16)
    amax = np.max(np.abs(wg), axis=1)
    s = codecs.e4m3(amax / (6.0 * t))
    sb = codecs.encode_e4m3(s)
    denom = s * t                                  # exact: two short significands
    scaled = wg / np.where(denom > 0, denom, 1.0)[:, None, :]
    codes = codecs.encode_e2m1(scaled)
    codes = np.where((denom > 0)[:, None, :], codes, 0)
    return codes.reshape(w.shape).astype(np.uint8), sb.astype(np.uint8), t


# ------------------------------------------------------------ dequantization

def dequant_int(q, s, z, g: int, adt: str) -> np.ndarray:
    """w^[k, n] = adt((q[k,n] - z[k/g, n]) * s[k/g, n]), one rounding.

    ``z`` is None for symmetric INT4 (q already signed)."""
    q = np.asarray(q, dtype=np.float64)
    k, n = q.shape
    s_full = np.repeat(np.asarray(s, dtype=np.float64), g, axis=0)
    zz = 0.0 if z is None else np.repeat(np.asarray(z, dtype=np.float64), g, axis=0)
    exact = (q - zz) * s_full
    return codecs.round_dtype(adt)(exact)


def dequant_int_unrounded(q, s, z, g: int) -> np.ndarray:
    """(q - z) * s in float64 without the activation-dtype rounding (for
    reporting the alternative reading's error only)."""
    q = np.asarray(q, dtype=np.float64)
    s_full = np.repeat(np.asarray(s, dtype=np.float64), g, axis=0)
    zz = 0.0 if z is None else np.repeat(np.asarray(z, dtype=np.float64), g, axis=0)
    return (q - zz) * s_full


def dequant_mxfp4(codes, b) -> np.ndarray:
    """w^[k, n] = e2m1(codes[k, n]) * 2^(b[k/32, n] - 127), exact."""
    vals = codecs.decode_e2m1(codes)
    scale = np.repeat(codecs.decode_e8m0(b), 32, axis=0)
    return vals * scale


# ------------------------------------------------------------ standard format

def nvfp4_operand(codes, sb) -> np.ndarray:
    """e2m1(codes[k, n]) * e4m3(sb[k/16, n]): the exact value the kernels feed
    to the tensor core (the tensor scale multiplies the fp32 sum)."""
    return codecs.decode_e2m1(codes) * np.repeat(codecs.decode_e4m3(sb), 16, axis=0)


def dequant_nvfp4(codes, sb, t: float) -> np.ndarray:
    """w^[k, n] = e2m1(codes[k, n]) * e4m3(sb[k/16, n]) * t, exact in float64."""
    return nvfp4_operand(codes, sb) * float(t)


def pack_int4_kn(q, signed: bool) -> np.ndarray:
    """Codes [K, N] -> qweight int32 [K/8, N], k = 8j + i in bits [4i, 4i+4)."""
    q = np.asarray(q, dtype=np.int64)
    k, n = q.shape
    if k % 8:
        raise ValueError("K must be a multiple of 8")
    lo, hi = (-8, 7) if signed else (0, 15)
    if q.min(initial=lo) < lo or q.max(initial=hi) > hi:
        raise ValueError("code out of range")
    nib = (q & 0xF).astype(np.uint64).reshape(k // 8, 8, n)
    word = np.zeros((k // 8, n), dtype=np.uint64)
    for i in range(8):
        word |= nib[:, i, :] << np.uint64(4 * i)
    return word.astype(np.uint32).view(np.int32)


def unpack_int4_kn(qweight, signed: bool) -> np.ndarray:
    """Inverse of ``pack_int4_kn``."""
    w = np.asarray(qweight).view(np.uint32).astype(np.uint64)
    kw, n = w.shape
    out = np.empty((kw, 8, n), dtype=np.int64)
    for i in range(8):
        out[:, i, :] = (w >> np.uint64(4 * i)) & np.uint64(0xF)
    out = out.reshape(kw * 8, n)
    if signed:
        out = np.where(out >= 8, out - 16, out)
    return out


def pack_zeros(z) -> np.ndarray:
    """Zeros [K/g, N] in [0,15] -> qzeros int32 [K/g, N/8], column 8j + i in
    nibble i of word (G, j)."""
    z = np.asarray(z, dtype=np.int64)
    gk, n = z.shape
    if n % 8:
        raise ValueError("N must be a multiple of 8")
    nib = (z & 0xF).astype(np.uint64).reshape(gk, n // 8, 8)
    word = np.zeros((gk, n // 8), dtype=np.uint64)
    for i in range(8):
        word |= nib[:, :, i] << np.uint64(4 * i)
    return word.astype(np.uint32).view(np.int32)


def unpack_zeros(qzeros) -> np.ndarray:
    w = np.asarray(qzeros).view(np.uint32).astype(np.uint64)
    gk, nw = w.shape
    out = np.empty((gk, nw, 8), dtype=np.int64)
    for i in range(8):
        out[:, :, i] = (w >> np.uint64(4 * i)) & np.uint64(0xF)
    return out.reshape(gk, nw * 8)


def pack_bits(v, bits: int) -> np.ndarray:
    """Codes v [L, ...] (as raw b-bit patterns, 0 <= v < 2^b) -> int32 words
    [L*b/32, ...]: code i of the stream occupies bits [b*i, b*i + b) of the
    little-endian concatenation of the words (a code may straddle two)."""
    v = np.asarray(v, dtype=np.int64)
    if (v.shape[0] * bits) % 32:
        raise ValueError("the stream must fill whole words")
    if v.min(initial=0) < 0 or v.max(initial=0) >= 2 ** bits:
        raise ValueError("code out of range")
    words = np.zeros((v.shape[0] * bits // 32,) + v.shape[1:], dtype=np.uint64)
    for i in range(v.shape[0]):
        bit = bits * i
        wi, off = bit // 32, bit % 32
        x = v[i].astype(np.uint64)
        words[wi] |= (x << np.uint64(off)) & np.uint64(0xFFFFFFFF)
        if off + bits > 32:
            words[wi + 1] |= x >> np.uint64(32 - off)
    return words.astype(np.uint32).view(np.int32)


def unpack_bits(words, bits: int) -> np.ndarray:
    """Inverse of ``pack_bits``: int32 words [W, ...] -> codes [32*W/b, ...]."""
    w = np.asarray(words).view(np.uint32).astype(np.uint64)
    count = w.shape[0] * 32 // bits
    out = np.empty((count,) + w.shape[1:], dtype=np.int64)
    mask = np.uint64(2 ** bits - 1)
    for i in range(count):
        bit = bits * i
        wi, off = bit // 32, bit % 32
        x = w[wi] >> np.uint64(off)
        if off + bits > 32:
            x |= w[wi + 1] << np.uint64(32 - off)
        out[i] = (x & mask).astype(np.int64)
    return out


def pack_int_kn(q, bits: int, signed: bool) -> np.ndarray:
    """Codes [K, N] of b bits -> qweight int32 [K*b/32, N] (b = 8: four codes
    a word; b = 3: 32 codes in three words), two's complement when signed."""
    q = np.asarray(q, dtype=np.int64)
    lo, hi = (-(2 ** (bits - 1)), 2 ** (bits - 1) - 1) if signed else (0, 2 ** bits - 1)
    if q.min(initial=lo) < lo or q.max(initial=hi) > hi:
        raise ValueError("code out of range")
    return pack_bits(q & (2 ** bits - 1), bits)


def unpack_int_kn(qweight, bits: int, signed: bool) -> np.ndarray:
    """Inverse of ``pack_int_kn``."""
    out = unpack_bits(qweight, bits)
    if signed:
        out = np.where(out >= 2 ** (bits - 1), out - 2 ** bits, out)
    return out


def pack_zeros_bits(z, bits: int) -> np.ndarray:
    """Zeros [K/g, N] of b bits -> qzeros int32 [K/g, N*b/32], packed along N
    like ``pack_bits`` (b = 4 gives ``pack_zeros``)."""
    return np.ascontiguousarray(pack_bits(np.asarray(z).T, bits).T)


def unpack_zeros_bits(qzeros, bits: int) -> np.ndarray:
    return np.ascontiguousarray(unpack_bits(np.asarray(qzeros).T, bits).T)


def pack_mxfp4(codes_kn, b_kn):
    """MXFP4 codes [K, N] and exponents [K/32, N] -> (uint8 [N, K/2] with the
    even k in the low nibble, uint8 [N, K/32])."""
    c = np.asarray(codes_kn, dtype=np.uint8).T          # [N, K]
    packed = (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)
    return (np.ascontiguousarray(packed, dtype=np.uint8),
            np.ascontiguousarray(np.asarray(b_kn, dtype=np.uint8).T))


def unpack_mxfp4(packed_nk, b_nk):
    """Inverse of ``pack_mxfp4``: -> (codes [K, N], b [K/32, N])."""
    p = np.asarray(packed_nk, dtype=np.uint8)
    n, kh = p.shape
    c = np.empty((n, 2 * kh), dtype=np.uint8)
    c[:, 0::2] = p & 0xF
    c[:, 1::2] = p >> 4
    return np.ascontiguousarray(c.T), np.ascontiguousarray(np.asarray(b_nk, dtype=np.uint8).T)


def pack_nvfp4(codes_kn, sb_kn):
    """NVFP4 codes [K, N] and e4m3 scales [K/16, N] -> (uint8 [N, K/2] with the
    even k in the low nibble, uint8 [N, K/16])."""
    c = np.asarray(codes_kn, dtype=np.uint8).T
    packed = (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)
    return np.ascontiguousarray(packed.astype(np.uint8)), np.ascontiguousarray(
        np.asarray(sb_kn, dtype=np.uint8).T)


def unpack_nvfp4(packed_nk, sb_nk):
    """Inverse of ``pack_nvfp4``: -> (codes [K, N], sb [K/16, N])."""
    p = np.asarray(packed_nk, dtype=np.uint8)
    n, kh = p.shape
    codes = np.empty((n, 2 * kh), dtype=np.uint8)
    codes[:, 0::2] = p & 0xF
    codes[:, 1::2] = p >> 4
    return codes.T.copy(), np.asarray(sb_nk, dtype=np.uint8).T.copy()


def scales_bits(s, sdt: str) -> np.ndarray:
    """Scale values -> uint16 bit patterns of the scale dtype."""
    return codecs.dtype_bits(sdt, s)
