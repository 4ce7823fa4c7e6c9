"""The kernel-side ("repacked") weight layout, written from its specification.

The Humming preprocessing step "checks parameters, pads dimensions and repacks
tensors for the target kernel" (kinachrichten.com, "Wie die Architektur
funktioniert"); the retrivium.ai retrospective ("Representation answers a
different question") adds that repacking may rearrange tensors for a device
without changing what the stored values mean.  The pages leave the target
layout to the implementation.  This module restates the layout that the CUDA
repack must produce, from the specification alone, so that the repack can be
checked bit for bit.

W4A16 tiled layout (N and K multiples of 128; KT = K / 128 k-tiles):

  weights: one 8192-byte block per (n-tile nt, k-tile kt), blocks ordered
    nt-major: block index nt * KT + kt.  A block is 512 little-endian 16-byte
    vectors; vector v = (qd * 4 + j) * 32 + t holds row n = 128 nt + 32 qd + t
    and the 32 values k = 128 kt + 32 j + [0, 32).  Its 32-bit word w
    (w = 0..3) holds k-offsets 8w + [0, 8) within the vector, nibble position
    p (bits [4p, 4p+4)) holding k-offset 8w + PERM[p] with
    PERM = [0, 2, 4, 6, 1, 3, 5, 7], so that nibbles p and p + 4 are the two
    consecutive k-offsets 8w + 2p and 8w + 2p + 1.
    Nibble value: offset binary q + 8 for signed INT4, the raw code for UINT4.

  scales: one block of 128 * ST 16-bit words per (nt, kt), same block order,
    with ST = max(1, 128 / g) groups touched by a k-tile; word sg * 128 + r is
    the scale of row n = 128 nt + r for the group holding
    k = 128 kt + sg * min(g, 128).

  zeros (UINT4 only): one block of 128 * ST bytes per (nt, kt), byte
    sg * 128 + r is the zero point (0..15) of the same (group, row).

INT8 / UINT8 tiled layout (W8A16; same tiling):

  weights: one 16384-byte block per (nt, kt); vector v = (qd * 8 + j) * 32 + t
    holds row n = 128 nt + 32 qd + t and the 16 values k = 128 kt + 16 j +
    [0, 16), byte c holding k-offset c.  Byte value: offset binary q + 128
    for signed INT8, the raw code for UINT8.
  scales, zeros: as W4A16 (zero points 0..255).

MXFP4 tiled layout (same tiling):

  weights: one 8192-byte block per (nt, kt), vector v = (qd * 4 + j) * 32 + t
    holds row n = 128 nt + 32 qd + t and k = 128 kt + 32 j + [0, 32) as 16
    bytes in the standard order (byte b: k = 2b in the low nibble, 2b + 1 in
    the high nibble), i.e. 32 consecutive codes of the row.
  scales: one 512-byte block per (nt, kt); bytes 4 r .. 4 r + 3 are the e8m0
    exponents of row n = 128 nt + r for k = 128 kt + [0, 32), [32, 64),
    [64, 96), [96, 128) in that order.

NVFP4 layout (same tiling; block size 8192 + 2048 bytes):

  weights: the MXFP4 code vectors above (32 consecutive codes of one row per
    16-byte vector, standard nibble order).
  scales: the W4A16 scale stream with g = 16 (ST = 8): word sg * 128 + r is
    the e4m3 block scale of row r for k = 128 kt + 16 sg .. + 15, written as
    the activation dtype's bit pattern (every e4m3 value is exact in bf16 and
    fp16, so this re-encodes without changing the value).
  tensor scales: after the last expert's blocks, one fp32 per expert, padded
    to a multiple of 16 bytes.

Gated layers (an MoE expert's gate|up projection, N = 2I: gate columns
[0, I), up columns [I, 2I)): the SiLU gate multiplies gate column i by up
column I + i, so the pack places the pair in one tile, on neighbouring rows:
row 2i + s of n-tile nt is standard column s * I + 64 nt + i (s = 0 gate,
s = 1 up).  The layout above then applies to the matrix with its columns in
that order.  The pages fix no pack order; this one is the implementation's.

Packed buffer (what the pack entry point writes): the three streams above
interleaved block by block, so that block (nt, kt) is one contiguous run of
bytes [weights block][scales block][zeros block] and the blocks follow in the
same nt-major order; experts follow one another, each expert's blocks
contiguous.  Block sizes: 8192 + 256 ST (+ 128 ST with zeros) bytes for
INT4/UINT4, 16384 + 256 ST (+ 128 ST) for INT8/UINT8, 8192 + 512 for MXFP4.
"""

from __future__ import annotations

import numpy as np

TILE_N = 128
TILE_K = 128
PERM = np.array([0, 2, 4, 6, 1, 3, 5, 7])


def scale_groups_per_tile(g: int) -> int:
    return max(1, TILE_K // g)


def tiled_weights(q, signed: bool) -> np.ndarray:
    """Codes q[K, N] -> the tiled byte stream (uint8, N*K/2 bytes)."""
    q = np.asarray(q, dtype=np.int64)
    k, n = q.shape
    nib = (q + 8) if signed else q.copy()
    if nib.min() < 0 or nib.max() > 15:
        raise ValueError("code out of range")
    kt_n, nt_n = k // TILE_K, n // TILE_N
    # nib4[kt, k_local, nt, n_local]
    nib4 = nib.astype(np.uint64).reshape(kt_n, TILE_K, nt_n, TILE_N)
    out = np.zeros((nt_n, kt_n, 4, 4, 32, 4), dtype=np.uint64)   # words
    for qd in range(4):
        for j in range(4):
            for w in range(4):
                for p in range(8):
                    kl = 32 * j + 8 * w + PERM[p]
                    vals = nib4[:, kl, :, 32 * qd: 32 * qd + 32]         # [KT, NT, 32]
                    out[:, :, qd, j, :, w] |= vals.transpose(1, 0, 2) << np.uint64(4 * p)
    return out.astype(np.uint32).reshape(-1).view(np.uint8)


def tiled_scales(s_bits, g: int, k: int) -> np.ndarray:
    """Scale bit patterns [K/g, N] (uint16) -> tiled uint16 stream."""
    s_bits = np.asarray(s_bits, dtype=np.uint16)
    n = s_bits.shape[1]
    st = scale_groups_per_tile(g)
    kt_n, nt_n = k // TILE_K, n // TILE_N
    out = np.zeros((nt_n, kt_n, st, TILE_N), dtype=np.uint16)
    for nt in range(nt_n):
        for kt in range(kt_n):
            for sg in range(st):
                kk = TILE_K * kt + sg * min(g, TILE_K)
                out[nt, kt, sg, :] = s_bits[kk // g, TILE_N * nt: TILE_N * (nt + 1)]
    return out.reshape(-1)


def tiled_weights8(q, signed: bool) -> np.ndarray:
    """8-bit codes q[K, N] -> the tiled byte stream (uint8, N*K bytes)."""
    q = np.asarray(q, dtype=np.int64)
    k, n = q.shape
    byte = (q + 128) if signed else q.copy()
    if byte.min() < 0 or byte.max() > 255:
        raise ValueError("code out of range")
    kt_n, nt_n = k // TILE_K, n // TILE_N
    out = np.zeros((nt_n, kt_n, 4, 8, 32, 16), dtype=np.uint8)   # [nt, kt, qd, j, t, c]
    for qd in range(4):
        for j in range(8):
            for c in range(16):
                kl = 16 * j + c
                rows = byte.reshape(kt_n, TILE_K, nt_n, TILE_N)[:, kl, :, 32 * qd: 32 * qd + 32]
                out[:, :, qd, j, :, c] = rows.transpose(1, 0, 2)
    return out.reshape(-1)


def tiled_zeros(z, g: int, k: int) -> np.ndarray:
    """Zero points [K/g, N] (0..15, or 0..255 for UINT8) -> tiled uint8 stream."""
    z = np.asarray(z, dtype=np.int64)
    n = z.shape[1]
    st = scale_groups_per_tile(g)
    kt_n, nt_n = k // TILE_K, n // TILE_N
    out = np.zeros((nt_n, kt_n, st, TILE_N), dtype=np.uint8)
    for nt in range(nt_n):
        for kt in range(kt_n):
            for sg in range(st):
                kk = TILE_K * kt + sg * min(g, TILE_K)
                out[nt, kt, sg, :] = z[kk // g, TILE_N * nt: TILE_N * (nt + 1)]
    return out.reshape(-1)


def tiled_weights_inverse(stream, k: int, n: int, signed: bool) -> np.ndarray:
    """Read the codes back out of a tiled stream (for round-trip checks)."""
    words = np.asarray(stream, dtype=np.uint8).view(np.uint32).astype(np.uint64)
    kt_n, nt_n = k // TILE_K, n // TILE_N
    words = words.reshape(nt_n, kt_n, 4, 4, 32, 4)
    q4 = np.full((kt_n, TILE_K, nt_n, TILE_N), -99, dtype=np.int64)
    for qd in range(4):
        for j in range(4):
            for w in range(4):
                for p in range(8):
                    kl = 32 * j + 8 * w + PERM[p]
                    vals = (words[:, :, qd, j, :, w] >> np.uint64(4 * p)) & np.uint64(0xF)
                    q4[:, kl, :, 32 * qd: 32 * qd + 32] = vals.transpose(1, 0, 2).astype(np.int64)
    q = q4.reshape(k, n)
    return q - 8 if signed else q


def tiled_mxfp4_weights(codes_nk) -> np.ndarray:
    """Standard MXFP4 codes uint8 [N, K/2] -> tiled byte stream."""
    c = np.asarray(codes_nk, dtype=np.uint8)
    n, kh = c.shape
    k = 2 * kh
    kt_n, nt_n = k // TILE_K, n // TILE_N
    # c4[nt, qd, t, kt, j, 16 bytes]
    c4 = c.reshape(nt_n, 4, 32, kt_n, 4, 16)
    out = c4.transpose(0, 3, 1, 4, 2, 5)          # nt, kt, qd, j, t, bytes
    return np.ascontiguousarray(out).reshape(-1)


def tiled_mxfp4_scales(b_nk) -> np.ndarray:
    """Standard e8m0 exponents uint8 [N, K/32] -> tiled byte stream."""
    b = np.asarray(b_nk, dtype=np.uint8)
    n, kb = b.shape
    kt_n, nt_n = kb // 4, n // TILE_N
    b4 = b.reshape(nt_n, TILE_N, kt_n, 4)
    return np.ascontiguousarray(b4.transpose(0, 2, 1, 3)).reshape(-1)


def glu_column_order(n: int) -> np.ndarray:
    """Standard column index held by each packed column of a gated layer of
    width n (gate half first): entry 128 nt + 2 i + s is s * n/2 + 64 nt + i."""
    if n % TILE_N:
        raise ValueError("n must be a multiple of 128")
    order = np.empty(n, dtype=np.int64)
    for nt in range(n // TILE_N):
        for i in range(TILE_N // 2):
            for s in range(2):
                order[TILE_N * nt + 2 * i + s] = s * (n // 2) + (TILE_N // 2) * nt + i
    return order


def glu_interleave_columns(x, axis: int = -1) -> np.ndarray:
    """x with its gate|up columns (along axis) in the gated pack order."""
    x = np.asarray(x)
    return np.take(x, glu_column_order(x.shape[axis]), axis=axis)


def interleave_blocks(*streams_and_sizes) -> np.ndarray:
    """Interleave per-block streams: arguments are (byte stream, block bytes)
    pairs with the same number of blocks; block i of the result is block i of
    each stream in argument order."""
    parts = []
    count = None
    for stream, size in streams_and_sizes:
        b = np.ascontiguousarray(stream).view(np.uint8).reshape(-1)
        if b.size % size:
            raise ValueError("stream is not a whole number of blocks")
        if count is None:
            count = b.size // size
        elif b.size // size != count:
            raise ValueError("streams hold different block counts")
        parts.append(b.reshape(count, size))
    return np.concatenate(parts, axis=1).reshape(-1)


def packed_w4(q, s_bits, z, g: int, signed: bool) -> np.ndarray:
    """Codes q[K, N], scale bits [K/g, N] and zero points [K/g, N] (None for
    signed INT4) -> the packed buffer of one matrix."""
    k = np.asarray(q).shape[0]
    st = scale_groups_per_tile(g)
    pieces = [(tiled_weights(q, signed), 8192), (tiled_scales(s_bits, g, k), 256 * st)]
    if z is not None:
        pieces.append((tiled_zeros(z, g, k), 128 * st))
    return interleave_blocks(*pieces)


def packed_w3(q, s_bits, z, g: int, signed: bool) -> np.ndarray:
    """The packed buffer of a 3-bit integer layer (GPTQ INT3 / UINT3).

    Reading (the pages name GPTQ INT3 among the served formats and fix no
    kernel layout): the 3-bit codes take the 4-bit blocks of ``packed_w4``
    unchanged in value.  An INT3 code q in [-4, 3] is a 4-bit two's
    complement value too, so it is stored as the offset-binary nibble q + 8
    like an INT4 code; a UINT3 code and its zero point (0..7) are stored as
    they are.  The dequantized value (q - z) * s is therefore the same in
    both representations."""
    q = np.asarray(q)
    lo, hi = (-4, 3) if signed else (0, 7)
    if q.min(initial=0) < lo or q.max(initial=0) > hi:
        raise ValueError("codes out of the 3-bit range")
    if z is not None and (np.asarray(z).min(initial=0) < 0 or np.asarray(z).max(initial=0) > 7):
        raise ValueError("zero points out of the 3-bit range")
    return packed_w4(q, s_bits, z, g, signed)


def packed_w8(q, s_bits, z, g: int, signed: bool) -> np.ndarray:
    """8-bit codes q[K, N], scale bits [K/g, N] and zero points [K/g, N] (None
    for signed INT8) -> the packed buffer of one matrix."""
    k = np.asarray(q).shape[0]
    st = scale_groups_per_tile(g)
    pieces = [(tiled_weights8(q, signed), 16384), (tiled_scales(s_bits, g, k), 256 * st)]
    if z is not None:
        pieces.append((tiled_zeros(z, g, k), 128 * st))
    return interleave_blocks(*pieces)


def packed_nvfp4(codes_nk, sb_nk, adt: str) -> np.ndarray:
    """Standard NVFP4 codes [N, K/2] and e4m3 scales [N, K/16] of one matrix ->
    its packed blocks (the tensor-scale tail is ``nvfp4_tail``)."""
    from . import codecs
    sb = np.asarray(sb_nk, dtype=np.uint8)
    k = sb.shape[1] * 16
    bits = codecs.dtype_bits(adt, codecs.decode_e4m3(sb)).T     # [K/16, N]
    return interleave_blocks((tiled_mxfp4_weights(codes_nk), 8192),
                             (tiled_scales(bits, 16, k), 2048))


def nvfp4_tail(tensor_scales) -> np.ndarray:
    """The per-expert fp32 tensor scales as bytes, padded to 16-byte multiples."""
    t = np.asarray(tensor_scales, dtype=np.float32).reshape(-1)
    pad = (-t.size) % 4
    return np.concatenate([t, np.zeros(pad, dtype=np.float32)]).view(np.uint8)


def packed_mxfp4(codes_nk, b_nk) -> np.ndarray:
    """Standard MXFP4 codes [N, K/2] and exponents [N, K/32] -> the packed
    buffer of one matrix."""
    return interleave_blocks((tiled_mxfp4_weights(codes_nk), 8192),
                             (tiled_mxfp4_scales(b_nk), 512))
