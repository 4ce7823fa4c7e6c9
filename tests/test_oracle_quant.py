"""Pins for the quantizers, the standard-format encoding, dequantization and
the kernel-side tiled layout."""

import numpy as np
import pytest

import synth
from conftest import read_golden
from oracle import codecs, layout, quant


def test_dequant_golden_cases():
    for row in read_golden("dequant_cases.txt"):
        if row[0] == "int":
            _, q, z, s, adt, want = row
            got = quant.dequant_int(np.array([[int(q)]]), np.array([[float(s)]]),
                                    np.array([[int(z)]]), 1, adt)
            assert float(got[0, 0]) == float(want), row
        elif row[0] == "mx":
            _, code, b, want = row
            got = quant.dequant_mxfp4(np.full((32, 1), int(code)), np.array([[int(b)]]))
            assert float(got[0, 0]) == float(want), row
        else:
            _, code, sbyte, t, want = row
            got = quant.dequant_nvfp4(np.full((16, 1), int(code)),
                                      np.array([[int(sbyte, 16)]]), float(t))
            assert float(got[0, 0]) == float(want), row


@pytest.mark.parametrize("sdt", ["fp16", "bf16"])
def test_int4_sym_invariants(sdt):
    g = synth.rng(5)
    w = synth.weights_fp32(g, 512, 64)
    q, s = quant.quantize_int4_sym(w, 128, sdt)
    assert q.min() >= -8 and q.max() <= 7
    assert np.array_equal(codecs.round_dtype(sdt)(s), s)          # s is representable
    full_s = np.repeat(s, 128, axis=0)
    err = np.abs(w.astype(np.float64) - q * full_s)
    inside = (q > -8) & (q < 7)
    assert np.all(err[inside] <= full_s[inside] / 2 * (1 + 1e-12))
    # the group's absmax element lands on +-7 (or -8 after scale rounding)
    wg = np.abs(w.astype(np.float64)).reshape(4, 128, 64)
    arg = wg.argmax(axis=1)
    qg = q.reshape(4, 128, 64)
    top = np.take_along_axis(qg, arg[:, None, :], axis=1)[:, 0, :]
    assert np.all(np.abs(top) >= 7)


def test_int4_sym_brute_force_small():
    g = synth.rng(6)
    w = synth.weights_fp32(g, 64, 8)
    q, s = quant.quantize_int4_sym(w, 32, "fp16")
    for gi in range(2):
        for n in range(8):
            col = [float(w[k, n]) for k in range(32 * gi, 32 * gi + 32)]
            amax = max(abs(v) for v in col)
            sv = float(np.float16(amax / 7.0))
            assert s[gi, n] == sv
            for i, v in enumerate(col):
                qq = max(-8, min(7, int(np.rint(v / sv))))
                assert q[32 * gi + i, n] == qq


def test_fp16_scales_with_bf16_activations_every_scale():
    """Every integer q - z in [-15, 15] against every finite fp16 scale: the
    oracle's one rounding to bf16 equals torch's round-to-nearest-even cast of
    the fp32 product (exact: 5 x 11 significant bits), and differs from
    rounding the scale to bf16 first on many of them."""
    import torch
    s16 = np.arange(1 << 16, dtype=np.uint16).view(np.float16)
    s16 = s16[np.isfinite(s16)].astype(np.float64)
    d = np.arange(-15, 16, dtype=np.float64)
    q = np.repeat(d[:, None], s16.size, axis=1)
    s = np.repeat(s16[None, :], d.size, axis=0)
    got = quant.dequant_int(q, s, None, 1, "bf16")
    prod = torch.from_numpy(q).float() * torch.from_numpy(s).float()
    want = prod.to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, want)
    pre = quant.dequant_int(q, codecs.round_dtype("bf16")(s), None, 1, "bf16")
    assert (pre != got).sum() > 1000


def test_int4_zero_group_scale_is_one():
    w = np.zeros((128, 8), dtype=np.float32)
    q, s = quant.quantize_int4_sym(w, 128, "bf16")
    assert np.all(s == 1.0) and np.all(q == 0)


def test_uint4_asym_invariants():
    g = synth.rng(7)
    w = synth.weights_fp32(g, 512, 64)
    q, s, z = quant.quantize_uint4_asym(w, 128, "bf16")
    assert q.min() >= 0 and q.max() <= 15 and z.min() >= 0 and z.max() <= 15
    full_s = np.repeat(s, 128, axis=0)
    full_z = np.repeat(z, 128, axis=0)
    err = np.abs(w.astype(np.float64) - (q - full_z) * full_s)
    inside = (q > 0) & (q < 15)
    assert np.all(err[inside] <= full_s[inside] / 2 * (1 + 1e-12))
    # the range spans all 16 codes up to rounding: min near 0, max near 15
    qg = q.reshape(4, 128, 64)
    assert np.all(qg.min(axis=1) <= 1) and np.all(qg.max(axis=1) >= 14)


def test_mxfp4_exponent_rule_and_codes():
    w = np.zeros((64, 3))
    w[:32, 0] = np.linspace(-6, 6, 32)                 # amax 6 -> E = 0, b = 127
    w[:32, 1] = 0.05 * np.linspace(-1, 1, 32)         # amax .05 -> floor(log2) = -5 -> E = -7
    w[32:, 2] = 0.0                                    # zero block -> b = 0, codes 0
    w[:32, 2] = 7.9                                    # saturates: E = 0, codes 6
    codes, b = quant.quantize_mxfp4(w)
    assert b[0, 0] == 127 and b[0, 1] == 120 and b[0, 2] == 127 and b[1, 2] == 0
    assert np.all(codecs.decode_e2m1(codes[:32, 2]) == 6.0)
    assert np.all(codes[32:, 2] == 0)
    deq = quant.dequant_mxfp4(codes, b)
    assert np.array_equal(deq[:32, 0], codecs.e2m1(w[:32, 0]))
    # relative error bound of e2m1 within the non-saturated range: half a step
    step = np.where(np.abs(w[:32, 1] / 2.0 ** -7) < 2, 0.5, np.where(np.abs(w[:32, 1] / 2.0 ** -7) < 4, 1.0, 2.0))
    assert np.all(np.abs(deq[:32, 1] - w[:32, 1]) <= step * 2.0 ** -7 / 2 + 1e-15)


def test_pack_unpack_roundtrip_and_handbuilt_words():
    g = np.random.default_rng(8)
    q = g.integers(-8, 8, (64, 40))
    assert np.array_equal(quant.unpack_int4_kn(quant.pack_int4_kn(q, True), True), q)
    u = g.integers(0, 16, (64, 40))
    assert np.array_equal(quant.unpack_int4_kn(quant.pack_int4_kn(u, False), False), u)
    # word 0x76543210 at (0, 0): k = 0..7 hold 0..7, least significant nibble first
    word = np.array([[0x76543210]], dtype=np.uint32).view(np.int32)
    assert list(quant.unpack_int4_kn(word, False)[:, 0]) == list(range(8))
    # signed: 0x89ABCDEF -> -1, -2, ..., -8
    word = np.array([[0x89ABCDEF]], dtype=np.uint32).view(np.int32)
    assert list(quant.unpack_int4_kn(word, True)[:, 0]) == [-1, -2, -3, -4, -5, -6, -7, -8]
    packed = quant.pack_int4_kn(np.arange(8).reshape(8, 1), False)
    assert packed.view(np.uint32)[0, 0] == 0x76543210


def test_zero_points_pack_handbuilt():
    z = np.arange(16).reshape(1, 16) % 16
    qz = quant.pack_zeros(z)
    assert qz.shape == (1, 2)
    assert qz.view(np.uint32)[0, 0] == 0x76543210 and qz.view(np.uint32)[0, 1] == 0xFEDCBA98
    assert np.array_equal(quant.unpack_zeros(qz), z)


def test_mxfp4_pack_handbuilt():
    codes = np.zeros((64, 2), dtype=np.uint8)
    codes[0, 0], codes[1, 0] = 1, 2           # k=0 low nibble, k=1 high nibble
    codes[63, 1] = 15
    b = np.full((2, 2), 127, dtype=np.uint8)
    b[1, 1] = 3
    p, bs = quant.pack_mxfp4(codes, b)
    assert p.flags.c_contiguous and bs.flags.c_contiguous
    assert p.shape == (2, 32) and p[0, 0] == 0x21 and p[1, 31] == 0xF0
    assert bs.shape == (2, 2) and bs[1, 1] == 3
    c2, b2 = quant.unpack_mxfp4(p, bs)
    assert np.array_equal(c2, codes) and np.array_equal(b2, b)


def _nibble_at(stream, n, k, kt_count):
    """Scalar statement of the tiled layout: location of (n, k)."""
    nt, nl = divmod(n, 128)
    kt, kl = divmod(k, 128)
    qd, t = divmod(nl, 32)
    j, r = divmod(kl, 32)
    w, o = divmod(r, 8)
    p = [0, 4, 1, 5, 2, 6, 3, 7][o]           # inverse of PERM: k-offset -> nibble position
    vec = (nt * kt_count + kt) * 512 + (qd * 4 + j) * 32 + t
    byte = vec * 16 + w * 4 + p // 2
    v = int(stream[byte])
    return (v >> 4) if p % 2 else (v & 0xF)


@pytest.mark.parametrize("signed", [True, False])
def test_tiled_layout_scalar_spec(signed):
    g = np.random.default_rng(9)
    k, n = 384, 256
    q = g.integers(-8, 8, (k, n)) if signed else g.integers(0, 16, (k, n))
    stream = layout.tiled_weights(q, signed)
    assert stream.size == k * n // 2
    for _ in range(3000):
        kk, nn = int(g.integers(0, k)), int(g.integers(0, n))
        want = q[kk, nn] + 8 if signed else q[kk, nn]
        assert _nibble_at(stream, nn, kk, k // 128) == want
    assert np.array_equal(layout.tiled_weights_inverse(stream, k, n, signed), q)


@pytest.mark.parametrize("gsize", [32, 64, 128, 256])
def test_tiled_scales_and_zeros_scalar_spec(gsize):
    g = np.random.default_rng(10)
    k, n = 512, 256
    sb = g.integers(0, 65535, (k // gsize, n)).astype(np.uint16)
    z = g.integers(0, 16, (k // gsize, n))
    ts = layout.tiled_scales(sb, gsize, k)
    tz = layout.tiled_zeros(z, gsize, k)
    st = max(1, 128 // gsize)
    assert ts.size == (k // 128) * (n // 128) * st * 128
    for kk in range(0, k, 32):
        for nn in range(0, n, 7):
            nt, r = divmod(nn, 128)
            kt, kl = divmod(kk, 128)
            sg = kl // gsize if gsize < 128 else 0
            idx = ((nt * (k // 128) + kt) * st + sg) * 128 + r
            assert ts[idx] == sb[kk // gsize, nn]
            assert tz[idx] == z[kk // gsize, nn]


def test_mxfp4_tiled_layout_scalar_spec():
    g = np.random.default_rng(14)
    n, k = 256, 384
    codes = g.integers(0, 256, (n, k // 2)).astype(np.uint8)
    b = g.integers(100, 140, (n, k // 32)).astype(np.uint8)
    ws = layout.tiled_mxfp4_weights(codes)
    ss = layout.tiled_mxfp4_scales(b)
    assert ws.size == n * k // 2 and ss.size == n * k // 32
    kt_count = k // 128
    for _ in range(2000):
        nn, kk = int(g.integers(0, n)), int(g.integers(0, k))
        nt, nl = divmod(nn, 128)
        kt, kl = divmod(kk, 128)
        qd, t = divmod(nl, 32)
        j, r = divmod(kl, 32)
        vec = (nt * kt_count + kt) * 512 + (qd * 4 + j) * 32 + t
        byte = int(ws[vec * 16 + r // 2])
        nib = (byte >> 4) if r % 2 else (byte & 0xF)
        sb = int(codes[nn, kk // 2])
        assert nib == ((sb >> 4) if kk % 2 else (sb & 0xF))
        assert ss[(nt * kt_count + kt) * 512 + nl * 4 + kl // 32] == b[nn, kk // 32]


@pytest.mark.parametrize("gsize,zp", [(32, True), (128, False), (256, True)])
def test_packed_buffer_scalar_spec(gsize, zp):
    """Each packed block is [codes 8192][scales 256 ST][zeros 128 ST], blocks
    in n-tile-major order: read single entries back by their byte address."""
    g = np.random.default_rng(17)
    k, n = 512, 256
    q = g.integers(0, 16, (k, n)) if zp else g.integers(-8, 8, (k, n))
    sb = g.integers(0, 65535, (k // gsize, n)).astype(np.uint16)
    z = g.integers(0, 16, (k // gsize, n)) if zp else None
    buf = layout.packed_w4(q, sb, z, gsize, signed=not zp)
    st = max(1, 128 // gsize)
    blk = 8192 + 256 * st + (128 * st if zp else 0)
    kt_count = k // 128
    assert buf.size == (k // 128) * (n // 128) * blk
    for _ in range(1500):
        kk, nn = int(g.integers(0, k)), int(g.integers(0, n))
        nt, r = divmod(nn, 128)
        kt, kl = divmod(kk, 128)
        base = (nt * kt_count + kt) * blk
        codes = buf[base: base + 8192]
        want = q[kk, nn] if zp else q[kk, nn] + 8
        # the block's codes sit at the start, so a one-block stream reader applies
        assert _nibble_at(codes, r, kl, 1) == want
        sg = kl // gsize if gsize < 128 else 0
        sbyte = base + 8192 + 2 * (sg * 128 + r)
        assert int(buf[sbyte]) | (int(buf[sbyte + 1]) << 8) == sb[kk // gsize, nn]
        if zp:
            assert buf[base + 8192 + 256 * st + sg * 128 + r] == z[kk // gsize, nn]


def test_packed_mxfp4_scalar_spec():
    g = np.random.default_rng(18)
    n, k = 256, 384
    codes = g.integers(0, 256, (n, k // 2)).astype(np.uint8)
    b = g.integers(100, 140, (n, k // 32)).astype(np.uint8)
    buf = layout.packed_mxfp4(codes, b)
    kt_count = k // 128
    assert buf.size == (n // 128) * kt_count * (8192 + 512)
    for _ in range(1500):
        nn, kk = int(g.integers(0, n)), int(g.integers(0, k))
        nt, nl = divmod(nn, 128)
        kt, kl = divmod(kk, 128)
        qd, t = divmod(nl, 32)
        j, rr = divmod(kl, 32)
        base = (nt * kt_count + kt) * (8192 + 512)
        byte = int(buf[base + ((qd * 4 + j) * 32 + t) * 16 + rr // 2])
        nib = (byte >> 4) if rr % 2 else (byte & 0xF)
        assert nib == (codes[nn, kk // 2] >> (4 * (kk % 2))) & 0xF
        assert buf[base + 8192 + 4 * nl + j] == b[nn, kk // 32]


@pytest.mark.parametrize("n", [128, 384, 1024])
def test_glu_column_order_pairs_gate_with_up(n):
    """The gated pack order is a permutation in which every tile-row pair
    (2i, 2i+1) holds a gate column and its up column (n/2 apart), and each
    tile's gate columns are 64 consecutive output columns."""
    order = layout.glu_column_order(n)
    assert sorted(order.tolist()) == list(range(n))
    pairs = order.reshape(-1, 2)
    assert np.all(pairs[:, 0] < n // 2) and np.all(pairs[:, 1] - pairs[:, 0] == n // 2)
    gate_per_tile = pairs[:, 0].reshape(n // 128, 64)
    assert np.array_equal(gate_per_tile, np.arange(n // 2).reshape(n // 128, 64))


def test_glu_interleave_gives_the_same_gated_product():
    """Pairing neighbouring columns of the interleaved GU reproduces
    silu(G) * U of the standard layout exactly."""
    from oracle import moe
    g = np.random.default_rng(23)
    inter = 192
    gu = codecs.bf16(g.standard_normal((7, 2 * inter)) * 3)
    gi = layout.glu_interleave_columns(gu)
    paired = np.concatenate([gi[:, 0::2], gi[:, 1::2]], axis=1)   # [G | U] again
    assert np.array_equal(moe.silu_mul(paired, inter), moe.silu_mul(gu, inter))
    assert np.array_equal(paired, gu)


def test_gated_packed_buffer_scalar_spec():
    """Row 2i + s of n-tile nt of a gated layer's packed codes and scales holds
    standard column s * N/2 + 64 nt + i."""
    g = np.random.default_rng(24)
    k, n, gsize = 256, 384, 128
    q = g.integers(0, 16, (k, n))
    sb = g.integers(0, 65535, (k // gsize, n)).astype(np.uint16)
    z = g.integers(0, 16, (k // gsize, n))
    il = layout.glu_interleave_columns
    buf = layout.packed_w4(il(q), il(sb), il(z), gsize, signed=False)
    blk = 8192 + 256 + 128
    for _ in range(800):
        kk, nt, i, s = (int(g.integers(0, k)), int(g.integers(0, n // 128)),
                        int(g.integers(0, 64)), int(g.integers(0, 2)))
        src = s * (n // 2) + 64 * nt + i
        r = 2 * i + s
        kt, kl = divmod(kk, 128)
        base = (nt * (k // 128) + kt) * blk
        assert _nibble_at(buf[base: base + 8192], r, kl, 1) == q[kk, src]
        sbyte = base + 8192 + 2 * r
        assert int(buf[sbyte]) | (int(buf[sbyte + 1]) << 8) == sb[kk // gsize, src]
        assert buf[base + 8192 + 256 + r] == z[kk // gsize, src]


# ------------------------------------------------------------------ NVFP4

def test_nvfp4_round_trip_on_the_grid():
    """Weights built exactly on the NVFP4 grid (a +-6 element in every block,
    one block with scale 448 to fix the tensor scale) quantize back to the
    codes, scales and tensor scale they were built from."""
    g = np.random.default_rng(41)
    k, n = 128, 32
    t = 2.0 ** -7
    sb = g.choice(np.arange(0x08, 0x7F), size=(k // 16, n)).astype(np.uint8)   # normal e4m3
    sb[0, 0] = 0x7E                                                            # 448
    codes = g.integers(0, 16, (k, n)).astype(np.uint8)
    codes[0::16, :] = 7                                                        # +6 in each block
    w = quant.dequant_nvfp4(codes, sb, t)
    c2, sb2, t2 = quant.quantize_nvfp4(w)
    assert t2 == t
    assert np.array_equal(sb2, sb)
    # -0 and +0 decode alike; compare values
    assert np.array_equal(codecs.decode_e2m1(c2), codecs.decode_e2m1(codes))


def test_nvfp4_error_bound_and_ranges():
    """Random weights: codes and scales in range, block scales <= 448, and
    |w - w^| <= s * t (one grid unit of the block: e2m1's largest gap is 2)."""
    g = np.random.default_rng(42)
    w = g.standard_normal((512, 64)) * 0.03
    w[::7, 5] *= 40.0                                     # a few large outliers
    codes, sb, t = quant.quantize_nvfp4(w)
    assert codes.max() <= 15 and sb.max() <= 0x7E
    s = codecs.decode_e4m3(sb)
    assert np.all(s >= 0) and np.all(s <= 448)
    err = np.abs(w - quant.dequant_nvfp4(codes, sb, t))
    bound = np.repeat(s * t, 16, axis=0)
    assert np.all(err <= bound * (1 + 1e-12))
    assert t == float(np.float32(np.max(np.abs(w)) / 2688.0))


def test_nvfp4_zero_blocks_and_zero_matrix():
    w = np.zeros((32, 16))
    w[16:, 3] = 2688.0 * 2.0 ** -10          # t = 2^-10 exactly, s = 448, code 6
    codes, sb, t = quant.quantize_nvfp4(w)
    assert np.all(codes[:16] == 0) and np.all(sb[0] == 0)
    assert np.array_equal(quant.dequant_nvfp4(codes, sb, t), w)
    codes, sb, t = quant.quantize_nvfp4(np.zeros((16, 4)))
    assert t == 1.0 and not codes.any() and not sb.any()


def test_nvfp4_operand_is_exact_in_both_16_bit_types():
    """Every e2m1 x e4m3 product is a bf16 and an fp16 value (<= 5 significant
    bits, magnitude <= 2688, >= 2^-10): the kernel's dequant needs no rounding."""
    codes = np.repeat(np.arange(16, dtype=np.uint8), 16)[:, None]               # [256, 1]
    for sbyte in range(0x00, 0x7F):
        sb = np.full((16, 1), sbyte, dtype=np.uint8)
        v = quant.nvfp4_operand(codes, sb)
        codecs.bf16_bits(v)
        codecs.fp16_bits(v)


def test_nvfp4_brute_force_dequant():
    g = np.random.default_rng(43)
    codes = g.integers(0, 16, (32, 3)).astype(np.uint8)
    sb = g.integers(0, 0x7F, (2, 3)).astype(np.uint8)
    t = 0.375
    got = quant.dequant_nvfp4(codes, sb, t)
    for kk in range(32):
        for nn in range(3):
            c = int(codes[kk, nn])
            mag = [0, 0.5, 1, 1.5, 2, 3, 4, 6][c & 7]
            e4 = int(sb[kk // 16, nn])
            e, m = (e4 >> 3) & 15, e4 & 7
            sv = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
            want = (-mag if c & 8 else mag) * sv * t
            assert got[kk, nn] == want


def test_nvfp4_standard_pack_round_trip():
    g = np.random.default_rng(44)
    codes = g.integers(0, 16, (64, 8)).astype(np.uint8)
    sb = g.integers(0, 0x7F, (4, 8)).astype(np.uint8)
    cn, sn = quant.pack_nvfp4(codes, sb)
    assert cn.shape == (8, 32) and sn.shape == (8, 4)
    assert (cn[2, 5] & 0xF) == codes[10, 2] and (cn[2, 5] >> 4) == codes[11, 2]
    c2, s2 = quant.unpack_nvfp4(cn, sn)
    assert np.array_equal(c2, codes) and np.array_equal(s2, sb)


@pytest.mark.parametrize("adt", ["bf16", "fp16"])
def test_packed_nvfp4_scalar_spec(adt):
    """Block (nt, kt) is [codes 8192][scales 2048]: the codes as MXFP4's, the
    scale of (row r, 16-k group sg) at word sg * 128 + r in the activation
    dtype's bits; the tail holds the fp32 tensor scales."""
    g = np.random.default_rng(45)
    n, k = 256, 256
    codes = g.integers(0, 256, (n, k // 2)).astype(np.uint8)
    sb = g.integers(0, 0x7F, (n, k // 16)).astype(np.uint8)
    buf = layout.packed_nvfp4(codes, sb, adt)
    kt_count = k // 128
    assert buf.size == (n // 128) * kt_count * 10240
    for _ in range(1500):
        nn, kk = int(g.integers(0, n)), int(g.integers(0, k))
        nt, nl = divmod(nn, 128)
        kt, kl = divmod(kk, 128)
        qd, t = divmod(nl, 32)
        j, rr = divmod(kl, 32)
        base = (nt * kt_count + kt) * 10240
        byte = int(buf[base + ((qd * 4 + j) * 32 + t) * 16 + rr // 2])
        assert ((byte >> 4) if rr % 2 else (byte & 0xF)) == (codes[nn, kk // 2] >> (4 * (kk % 2))) & 0xF
        word = base + 8192 + 2 * ((kl // 16) * 128 + nl)
        bits = int(buf[word]) | (int(buf[word + 1]) << 8)
        assert codecs.dtype_from_bits(adt, np.array([bits]))[0] == codecs.decode_e4m3(sb[nn, kk // 16])
    tail = layout.nvfp4_tail([0.5, 2.0, -1.0])
    assert tail.size == 16 and list(tail.view(np.float32)) == [0.5, 2.0, -1.0, 0.0]


# ------------------------------------------------ other integer widths (8 and 3 bits)

def test_bitstream_handbuilt_words():
    # INT3: the codes 0..7 repeated over 32 k are the octal digits 76543210
    # (0xFAC688) four times over 96 bits, least significant code first:
    # 0xFAC688FAC688FAC688FAC688 -> words (low first) 88FAC688, C688FAC6, FAC688FA.
    q = np.tile(np.arange(8), 4)[:, None]
    words = quant.pack_int_kn(q, 3, signed=False)[:, 0].view(np.uint32)
    assert [int(x) for x in words] == [0x88FAC688, 0xC688FAC6, 0xFAC688FA]
    assert np.array_equal(quant.unpack_int_kn(words.view(np.int32)[:, None], 3, False), q)
    # signed INT3 -4..3 are the raw patterns 4, 5, 6, 7, 0, 1, 2, 3: octal
    # 32107654 = 0x688FAC per eight codes
    sq = np.tile(np.array([-4, -3, -2, -1, 0, 1, 2, 3]), 4)[:, None]
    sw = quant.pack_int_kn(sq, 3, signed=True)[:, 0].view(np.uint32)
    assert [int(x) for x in sw] == [0xAC688FAC, 0x8FAC688F, 0x688FAC68]
    assert np.array_equal(quant.unpack_int_kn(sw.view(np.int32)[:, None], 3, True), sq)
    # INT8: the bytes of k = 0..3, least significant first
    q8 = np.array([[0], [1], [127], [-128]])
    assert int(quant.pack_int_kn(q8, 8, signed=True)[0, 0].view(np.uint32)) == 0x807F0100
    assert int(quant.pack_int_kn(np.array([[1], [2], [3], [4]]), 8, False)[0, 0]) == 0x04030201
    # zeros pack along N the same way: a zero of 5 in 32 columns is the bit
    # pattern 101 repeated from bit 0 (nibbles D, 6, B, ...)
    zw = quant.pack_zeros_bits(np.full((1, 32), 5), 3)[0].view(np.uint32)
    assert [int(x) for x in zw] == [0x6DB6DB6D, 0xDB6DB6DB, 0xB6DB6DB6]


def test_bitstream_of_four_bits_is_the_nibble_layout():
    g = synth.rng(11)
    q = g.integers(-8, 8, size=(64, 24))
    assert np.array_equal(quant.pack_int_kn(q, 4, signed=True), quant.pack_int4_kn(q, True))
    z = g.integers(0, 16, size=(3, 32))
    assert np.array_equal(quant.pack_zeros_bits(z, 4), quant.pack_zeros(z))


@pytest.mark.parametrize("bits", [3, 8])
@pytest.mark.parametrize("signed", [True, False])
def test_bitstream_round_trip_every_code(bits, signed):
    lo = -(2 ** (bits - 1)) if signed else 0
    k = 32 * 2 ** bits // 8 if bits == 8 else 96
    g = synth.rng(12 + bits)
    q = (np.arange(k * 5).reshape(k, 5) % (2 ** bits)) + lo
    q = g.permuted(q, axis=0)
    words = quant.pack_int_kn(q, bits, signed)
    assert words.shape == (k * bits // 32, 5) and words.dtype == np.int32
    assert np.array_equal(quant.unpack_int_kn(words, bits, signed), q)
    z = g.integers(0, 2 ** bits, size=(4, 64))
    assert np.array_equal(quant.unpack_zeros_bits(quant.pack_zeros_bits(z, bits), bits), z)
    too_big = 2 ** (bits - 1) if signed else 2 ** bits     # one past the largest code
    with pytest.raises(ValueError):
        quant.pack_int_kn(np.full((k, 1), too_big), bits, signed)


def test_four_bit_quantizers_are_the_int4_ones():
    g = synth.rng(13)
    w = synth.weights_fp32(g, 256, 16)
    q, s = quant.quantize_int_sym(w, 64, "bf16", 4)
    q4, s4 = quant.quantize_int4_sym(w, 64, "bf16")
    assert np.array_equal(q, q4) and np.array_equal(s, s4)
    q, s, z = quant.quantize_uint_asym(w, 64, "fp16", 4)
    q4, s4, z4 = quant.quantize_uint4_asym(w, 64, "fp16")
    assert np.array_equal(q, q4) and np.array_equal(s, s4) and np.array_equal(z, z4)


@pytest.mark.parametrize("bits", [3, 8])
def test_int_quantizer_invariants(bits):
    g = synth.rng(14 + bits)
    w = synth.weights_fp32(g, 512, 48)
    top = 2 ** (bits - 1) - 1
    q, s = quant.quantize_int_sym(w, 128, "fp16", bits)
    assert q.min() >= -top - 1 and q.max() <= top
    assert np.array_equal(codecs.round_dtype("fp16")(s), s)
    full = np.repeat(s, 128, axis=0)
    err = np.abs(w.astype(np.float64) - q * full)
    inside = (q > -top - 1) & (q < top)
    assert np.all(err[inside] <= full[inside] / 2 * (1 + 1e-12))
    arg = np.abs(w.astype(np.float64)).reshape(4, 128, 48).argmax(axis=1)
    peak = np.take_along_axis(q.reshape(4, 128, 48), arg[:, None, :], axis=1)[:, 0, :]
    assert np.all(np.abs(peak) >= top)
    q, s, z = quant.quantize_uint_asym(w, 128, "bf16", bits)
    assert q.min() >= 0 and q.max() <= 2 ** bits - 1 and z.min() >= 0 and z.max() <= 2 ** bits - 1
    full_z = np.repeat(z, 128, axis=0)
    full = np.repeat(s, 128, axis=0)
    err = np.abs(w.astype(np.float64) - (q - full_z) * full)
    inside = (q > 0) & (q < 2 ** bits - 1)
    assert np.all(err[inside] <= full[inside] / 2 * (1 + 1e-12))


def test_int8_sym_brute_force_small():
    g = synth.rng(15)
    w = synth.weights_fp32(g, 64, 4)
    q, s = quant.quantize_int_sym(w, 32, "bf16", 8)
    for gi in range(2):
        for n in range(4):
            col = [float(w[k, n]) for k in range(32 * gi, 32 * gi + 32)]
            sv = float(codecs.bf16(np.array(max(abs(v) for v in col) / 127.0)))
            assert s[gi, n] == sv
            for i, v in enumerate(col):
                assert q[32 * gi + i, n] == max(-128, min(127, int(np.rint(v / sv))))


@pytest.mark.parametrize("gsize,zp", [(32, True), (128, False), (256, True)])
def test_packed_w8_scalar_spec(gsize, zp):
    """8-bit packed blocks are [codes 16384][scales 256 ST][zeros 128 ST]: the
    byte of (k, n) is byte 16 v + c of its block with v = (qd*8 + j)*32 + t,
    row 32 qd + t, k-offset 16 j + c; read single entries back by address."""
    g = np.random.default_rng(18)
    k, n = 512, 256
    q = g.integers(0, 256, (k, n)) if zp else g.integers(-128, 128, (k, n))
    sb = g.integers(0, 65535, (k // gsize, n)).astype(np.uint16)
    z = g.integers(0, 256, (k // gsize, n)) if zp else None
    buf = layout.packed_w8(q, sb, z, gsize, signed=not zp)
    st = max(1, 128 // gsize)
    blk = 16384 + 256 * st + (128 * st if zp else 0)
    kt_count = k // 128
    assert buf.size == kt_count * (n // 128) * blk
    for _ in range(1500):
        kk, nn = int(g.integers(0, k)), int(g.integers(0, n))
        nt, r = divmod(nn, 128)
        kt, kl = divmod(kk, 128)
        base = (nt * kt_count + kt) * blk
        qd, t = divmod(r, 32)
        j, c = divmod(kl, 16)
        v = (qd * 8 + j) * 32 + t
        assert buf[base + 16 * v + c] == (q[kk, nn] if zp else q[kk, nn] + 128)
        sg = kl // gsize if gsize < 128 else 0
        sbyte = base + 16384 + 2 * (sg * 128 + r)
        assert int(buf[sbyte]) | (int(buf[sbyte + 1]) << 8) == sb[kk // gsize, nn]
        if zp:
            assert buf[base + 16384 + 256 * st + sg * 128 + r] == z[kk // gsize, nn]


@pytest.mark.parametrize("zp", [False, True])
def test_packed_w3_scalar_spec(zp):
    """3-bit codes in the 4-bit blocks: an INT3 code q reads back as the
    nibble q + 8 and a UINT3 code (and its zero point) as itself, at the byte
    addresses of the 4-bit layout; codes from the standard bit stream."""
    g = np.random.default_rng(31)
    k, n, gsize = 256, 256, 64
    q = g.integers(0, 8, (k, n)) if zp else g.integers(-4, 4, (k, n))
    # through the standard format (bit stream along K) and back
    q = quant.unpack_int_kn(quant.pack_int_kn(q, 3, not zp), 3, not zp)
    sb = g.integers(0, 65535, (k // gsize, n)).astype(np.uint16)
    z = g.integers(0, 8, (k // gsize, n)) if zp else None
    buf = layout.packed_w3(q, sb, z, gsize, signed=not zp)
    st = 128 // gsize
    blk = 8192 + 256 * st + (128 * st if zp else 0)
    for _ in range(1500):
        kk, nn = int(g.integers(0, k)), int(g.integers(0, n))
        nt, r = divmod(nn, 128)
        kt, kl = divmod(kk, 128)
        base = (nt * (k // 128) + kt) * blk
        want = q[kk, nn] if zp else q[kk, nn] + 8
        assert _nibble_at(buf[base: base + 8192], r, kl, 1) == want
        if zp:
            assert buf[base + 8192 + 256 * st + (kl // gsize) * 128 + r] == z[kk // gsize, nn]


def test_packed_w3_rejects_codes_out_of_range():
    q = np.zeros((128, 128), dtype=np.int64)
    sb = np.zeros((1, 128), dtype=np.uint16)
    q[5, 7] = -5
    with pytest.raises(ValueError):
        layout.packed_w3(q, sb, None, 128, signed=True)
    q[5, 7] = 8
    with pytest.raises(ValueError):
        layout.packed_w3(q, sb, np.zeros((1, 128), dtype=np.int64), 128, signed=False)
