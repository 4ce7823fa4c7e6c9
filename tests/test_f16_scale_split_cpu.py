"""The arithmetic behind the kernels' dequantization of fp16 scales against
bf16 activations, checked over every finite fp16 scale and every integer
d = q - z in [-15, 15]: the scale splits into s_hi (its leading 8 significant
bits) and s_lo = s - s_hi, both bf16 values, s_lo with the sign of s (or a
zero of that sign); d * s_lo is exact in bf16; and one rounding of
d * s_hi + d * s_lo (a fused multiply-add) is the one rounding of d * s,
bit for bit including the sign of zero results."""

import numpy as np
import torch


def _split(s32):
    sb = s32.view(np.uint32)
    hi = (sb & 0xFFFF0000).view(np.float32)
    rest = s32 - hi
    lo = (((rest.view(np.uint32) >> 16) | ((sb >> 16) & 0x8000)) << 16).astype(np.uint32)
    return hi, rest, lo.view(np.float32)


def _bf16_bits(x64):
    # x64 holds values exact in fp32; the cast to bf16 rounds once
    return torch.from_numpy(x64).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy()


def test_split_terms_are_bf16_values():
    s16 = np.arange(1 << 16, dtype=np.uint16).view(np.float16)
    s = s16[np.isfinite(s16)].astype(np.float32)
    hi, rest, lo = _split(s)
    assert np.all((hi.view(np.uint32) & 0xFFFF) == 0)
    assert np.all((rest.view(np.uint32) & 0xFFFF) == 0)          # exact in bf16
    assert np.all(hi.astype(np.float64) + rest == s)               # nothing lost
    assert np.all(np.signbit(lo) == np.signbit(s))
    assert np.all(np.abs(rest) < np.abs(s) * 2.0 ** -7 + 1e-45)


def test_one_fma_rounds_the_exact_product_once():
    s16 = np.arange(1 << 16, dtype=np.uint16).view(np.float16)
    s = s16[np.isfinite(s16)].astype(np.float32)
    hi, _, lo = _split(s)
    hi64, lo64, s64 = hi.astype(np.float64), lo.astype(np.float64), s.astype(np.float64)
    for d in range(-15, 16):
        t = d * lo64
        assert np.array_equal(torch.from_numpy(t).to(torch.bfloat16).double().numpy(), t)
        assert np.array_equal(_bf16_bits(d * hi64 + t), _bf16_bits(d * s64)), d
