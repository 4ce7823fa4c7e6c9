"""Pins of the oracle's NVFP4 activation quantizer and W4A4 reference
(NVFP4 weights and activations; the pages list W4A4 among the common
configurations and name NVFP4: kinachrichten.com, "Warum quantisierte Kernel
wichtig sind").  Each check is independent of the oracle's own code: the
formats' values are written out here from their definitions (OCP FP4 e2m1 and
FP8 e4m3), nearest values are found by exhaustive search rather than by
rounding arithmetic, and the GEMM is summed in plain Python loops."""

import itertools

import numpy as np
import pytest

from oracle import gemm

# e2m1 magnitudes of codes 0..7: 0, subnormal 0.5, then (1 + m/2) 2^(e-1)
E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
# e4m3 magnitudes of bytes 0..126 (127 is NaN): subnormal m/8 2^-6, else (1 + m/8) 2^(e-7)
E4M3_MAG = [(m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
            for e in range(16) for m in range(8)][:127]


def _nearest_even(v, table):
    """Index of the table value nearest v (v >= 0), ties to the even index,
    saturating at the last entry: found by scanning every entry."""
    best = None
    for i, t in enumerate(table):
        d = abs(v - t)
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def _brute_quant(x, a_ts):
    m, k = x.shape
    codes = np.zeros((m, k), dtype=np.uint8)
    sb = np.zeros((m, k // 16), dtype=np.uint8)
    f = np.float32
    for r in range(m):
        for b in range(k // 16):
            blk = [f(v) for v in x[r, 16 * b:16 * b + 16]]
            amax = max(abs(v) for v in blk)
            t = f(amax / f(f(6.0) * f(a_ts)))
            si = _nearest_even(float(t), E4M3_MAG)
            sb[r, b] = si
            den = f(f(E4M3_MAG[si]) * f(a_ts))
            for j, v in enumerate(blk):
                if den == 0:
                    continue
                q = f(v / den)
                c = _nearest_even(abs(float(q)), E2M1_MAG)
                codes[r, 16 * b + j] = c | (8 if np.signbit(q) else 0)
    return codes, sb


def _bf16_values(g, shape, scale):
    x = (g.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("a_ts", [1.0, 2.0 ** -7, 0.0123, 3.5])
def test_act_quant_matches_exhaustive_search(a_ts):
    g = np.random.default_rng(5)
    x = _bf16_values(g, (3, 64), 1.0)
    x[0, 5] = 0.0
    x[1, 16:32] *= 1e-4                   # a block of small values
    x[2, 32:48] = 0.0                     # an all-zero block
    codes, sb = gemm.act_quant_nvfp4(x, a_ts)
    want_c, want_s = _brute_quant(x, a_ts)
    assert np.array_equal(sb, want_s)
    assert np.array_equal(codes, want_c)


def test_act_quant_round_trips_grid_values():
    """Blocks built from grid values whose largest magnitude is 6 come back
    unchanged: amax / (6 a_ts) is the block scale itself, every x / (s a_ts)
    a code value."""
    g = np.random.default_rng(6)
    a_ts = 0.125
    m, k = 4, 128
    codes = g.integers(0, 16, size=(m, k)).astype(np.uint8)
    codes[codes == 8] = 0                 # no negative zero
    codes[:, ::16] = 7                    # +6 in every block
    sbytes = g.integers(0x08, 0x70, size=(m, k // 16)).astype(np.uint8)
    val = np.array([E2M1_MAG[c & 7] * (-1 if c & 8 else 1) for c in codes.ravel()]).reshape(m, k)
    x = val * np.repeat([[E4M3_MAG[b] for b in row] for row in sbytes], 16, axis=1) * a_ts
    got_c, got_s = gemm.act_quant_nvfp4(x, a_ts)
    assert np.array_equal(got_s, sbytes)
    assert np.array_equal(got_c, codes)


def test_act_quant_special_blocks():
    a_ts = 1.0 / 64
    x = np.zeros((1, 48))
    x[0, 16:32] = 1e6 * np.linspace(-1, 1, 16)      # amax / (6 a_ts) far above 448
    x[0, 32] = -0.25 * a_ts * 2.0 ** -9               # tiny: t rounds to e4m3 zero
    codes, sb = gemm.act_quant_nvfp4(x, a_ts)
    assert sb[0, 0] == 0 and not codes[0, :16].any()  # zero block: scale 0, codes 0
    assert sb[0, 1] == 0x7E                            # saturated at 448
    assert codes[0, 16] == 0xF and codes[0, 31] == 0x7  # -6 and +6
    assert sb[0, 2] == 0 and not codes[0, 32:].any()


def test_w4a4_reference_equals_loop_sum():
    g = np.random.default_rng(7)
    m, k, n = 3, 32, 5
    ac = g.integers(0, 16, size=(m, k)).astype(np.uint8)
    asb = g.integers(0x20, 0x50, size=(m, k // 16)).astype(np.uint8)
    wc = g.integers(0, 16, size=(k, n)).astype(np.uint8)
    wsb = g.integers(0x20, 0x50, size=(k // 16, n)).astype(np.uint8)
    a_ts, w_ts = 0.5, 0.03125
    bias = g.standard_normal(n)
    got = gemm.w4a4_reference(ac, asb, a_ts, wc, wsb, w_ts, bias)

    def val(c, s):
        return E2M1_MAG[c & 7] * (-1 if c & 8 else 1) * E4M3_MAG[s]

    for i, j in itertools.product(range(m), range(n)):
        acc = sum(val(ac[i, kk], asb[i, kk // 16]) * val(wc[kk, j], wsb[kk // 16, j])
                  for kk in range(k))
        assert got[i, j] == pytest.approx(acc * a_ts * w_ts + bias[j], rel=1e-14, abs=1e-14)


def test_w4a4_reference_of_quantized_inputs_tracks_the_float_product():
    """End to end: quantizing both operands with NVFP4 keeps A W within the
    format's error (e2m1 keeps 2 significant bits: each operand's relative
    error is at most 1/4 per element, most far less)."""
    from oracle import quant
    g = np.random.default_rng(8)
    m, k, n = 8, 256, 16
    x = _bf16_values(g, (m, k), 1.0)
    w = g.standard_normal((k, n))
    wc, wsb, w_ts = quant.quantize_nvfp4(w)
    a_ts = float(np.max(np.abs(x))) / (6 * 448)
    ac, asb = gemm.act_quant_nvfp4(x, a_ts)
    got = gemm.w4a4_reference(ac, asb, a_ts, wc, wsb, w_ts)
    ref = x @ w
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 0.2


def _f32_neighbours(v, n=3):
    c = np.float32(v)
    out = [c]
    lo = hi = c
    for _ in range(n):
        lo = np.nextafter(lo, np.float32(-np.inf))
        hi = np.nextafter(hi, np.float32(np.inf))
        out += [lo, hi]
    return out


def _bf16_down(v):
    return float((np.array([v], np.float32).view(np.uint32) & np.uint32(0xFFFF0000))
                 .view(np.float32)[0])


def _fp32_decides_cases():
    """Blocks on which fp32 arithmetic and exact arithmetic decide differently:
    (kind, x row of 16, a_ts), found by search with this file's own arithmetic.
    Scale cases: fp32(1 / d) lands exactly on a midpoint between e4m3
    neighbours while 1 / d itself lies on the odd side.  Code cases: with the
    block scale s, fp32(x / fp32(s a_ts)) lands exactly on a midpoint between
    e2m1 neighbours while x / (s a_ts) lies on the odd side (s = 1: the divide
    decides; s with four significant bits: the product s a_ts too)."""
    f = np.float32
    cases = []
    mids = [(E4M3_MAG[i] + E4M3_MAG[i + 1]) / 2 for i in range(56, 70)]
    for mu in mids:
        for d in _f32_neighbours(1.0 / mu):
            if f(f(1.0) / d) != f(mu) or 1.0 / float(d) == mu:
                continue
            if _nearest_even(1.0 / float(d), E4M3_MAG) == _nearest_even(mu, E4M3_MAG):
                continue
            for a in _f32_neighbours(float(d) / 6.0):
                if f(f(6.0) * a) == d:
                    x = np.full(16, 0.5)
                    x[3] = 1.0
                    cases.append(("scale", x, float(a)))
                    break
    for sv in [1.0, 1.125, 1.375, 1.875]:
        for mu in [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]:
            for x0 in [1.0, 1.5, 1.25, 0.75]:
                for a in _f32_neighbours(x0 / (mu * sv), 6):
                    den = f(f(sv) * a)
                    if f(f(x0) / den) != f(mu):
                        continue
                    exact = x0 / (sv * float(a))
                    if exact == mu or _nearest_even(exact, E2M1_MAG) == _nearest_even(mu, E2M1_MAG):
                        continue
                    amax = _bf16_down(6.0 * sv * float(a))
                    t = f(f(amax) / f(f(6.0) * a))
                    if E4M3_MAG[_nearest_even(float(t), E4M3_MAG)] != sv or x0 > amax:
                        continue
                    x = np.full(16, 0.0)
                    x[0], x[1] = amax, x0
                    cases.append(("code" if sv == 1.0 else "product", x, float(a)))
                    break
    return cases


def test_act_quant_decides_in_fp32():
    """The oracle's scale and code decisions follow fp32 arithmetic where it
    differs from exact arithmetic (the kernel's precision)."""
    cases = _fp32_decides_cases()
    kinds = {c[0] for c in cases}
    assert kinds == {"scale", "code", "product"}, kinds
    for kind, x, a_ts in cases:
        codes, sb = gemm.act_quant_nvfp4(x[None, :], a_ts)
        want_c, want_s = _brute_quant(x[None, :], a_ts)
        assert np.array_equal(sb, want_s), (kind, a_ts)
        assert np.array_equal(codes, want_c), (kind, a_ts)
