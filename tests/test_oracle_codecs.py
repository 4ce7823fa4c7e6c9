"""Pins for the oracle's number formats: exhaustive tables, a library decoder,
hand-derived rounding cases, and bit-pattern identities."""

import math

import numpy as np
import pytest
import torch

from conftest import parse_float, read_golden
from oracle import codecs


def test_e2m1_table_matches_spec_fixture():
    rows = read_golden("e2m1_values.txt")
    assert len(rows) == 16
    for code_s, val_s in rows:
        code, val = int(code_s), float(val_s)
        got = codecs.decode_e2m1(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val)
        if code not in (0, 8):
            assert codecs.encode_e2m1(val) == code


def test_e4m3_decode_all_codes_vs_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = codecs.decode_e4m3(np.arange(256))
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], got[fin])
    assert np.nanmax(got) == 448.0 and np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def test_e4m3_encode_vs_torch_in_range():
    g = np.random.default_rng(11)
    x = np.concatenate([g.standard_normal(20000) * 50, g.standard_normal(5000) * 0.01,
                        g.uniform(-448, 448, 5000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = codecs.encode_e4m3(x.astype(np.float64))
    assert np.array_equal(ref, got)


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    vals = codecs.decode_e4m3(codes)
    assert np.array_equal(codecs.encode_e4m3(vals), codes)


def test_e8m0_values():
    assert codecs.decode_e8m0(127) == 1.0
    assert codecs.decode_e8m0(0) == 2.0 ** -127
    assert codecs.decode_e8m0(254) == 2.0 ** 127
    assert codecs.decode_e8m0(120) == 2.0 ** -7
    assert np.isnan(codecs.decode_e8m0(255))


@pytest.mark.parametrize("fmt", ["bf16", "fp16", "e4m3", "e2m1"])
def test_golden_rounding_cases(fmt):
    fn = {"bf16": codecs.bf16, "fp16": codecs.fp16, "e4m3": codecs.e4m3, "e2m1": codecs.e2m1}[fmt]
    rows = [r for r in read_golden("rounding_cases.txt") if r[0] == fmt]
    assert rows
    for _, xin, want in rows:
        got = float(fn(parse_float(xin)))
        assert got == parse_float(want), (fmt, xin, got, want)


def test_bf16_vs_torch_from_float32():
    g = np.random.default_rng(12)
    x = np.concatenate([g.standard_normal(50000), g.standard_normal(5000) * 1e-38,
                        g.standard_normal(5000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy().astype(np.float64)
    got = codecs.bf16(x.astype(np.float64))
    assert np.array_equal(ref, got)


def test_bf16_all_bit_patterns_are_fixed_points():
    bits = np.arange(65536, dtype=np.uint32)
    vals = codecs.bf16_from_bits(bits)
    fin = np.isfinite(vals)
    assert np.array_equal(codecs.bf16(vals[fin]), vals[fin])
    # the bit encoder inverts the decoder (the sign of zero included)
    assert np.array_equal(codecs.bf16_bits(vals[fin]), bits[fin].astype(np.uint16))


def test_bf16_midpoints_tie_to_even():
    bits = np.arange(0x3F80, 0x4000, dtype=np.uint32)        # [1, 2)
    lo = codecs.bf16_from_bits(bits)
    hi = codecs.bf16_from_bits(bits + 1)
    mid = (lo + hi) / 2
    r = codecs.bf16(mid)
    even = np.where(bits % 2 == 0, lo, hi)
    assert np.array_equal(r, even)


def test_fp16_vs_numpy_direct_double_conversion():
    g = np.random.default_rng(13)
    x = np.concatenate([g.standard_normal(50000) * 100, g.standard_normal(5000) * 1e-6,
                        g.uniform(-70000, 70000, 5000)])
    ref = x.astype(np.float16).astype(np.float64)
    got = codecs.fp16(x)
    assert np.array_equal(ref, got)


def test_fp16_all_bit_patterns_roundtrip():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = codecs.fp16_from_bits(bits)
    fin = np.isfinite(vals)
    assert np.array_equal(codecs.fp16(vals[fin]), vals[fin])
    assert np.array_equal(codecs.fp16_bits(vals[fin]), bits[fin])


def test_e2m1_rounding_exhaustive_grid():
    # every quarter step in [-8, 8]: brute force nearest grid value, ties even
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    codes_even = {0: True, 0.5: False, 1: True, 1.5: False, 2: True, 3: False, 4: True, 6: False}
    for x in np.arange(-8, 8.001, 0.125):
        m = abs(x)
        d = np.abs(grid - min(m, 6.0))
        best = grid[d == d.min()]
        want = best[0] if best.size == 1 else [b for b in best if codes_even[b]][0]
        want = math.copysign(want, x)
        got = float(codecs.e2m1(x))
        assert got == want or (got == 0 and want == 0), (x, got, want)
