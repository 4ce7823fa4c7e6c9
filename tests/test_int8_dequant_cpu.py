"""The arithmetic behind the kernels' dequantization of 8-bit codes against
bf16 activations, emulated step by step in IEEE fp32 on the CPU: the code u
placed in byte 1 of the fp32 pattern 0x47000000 reads 2^15 + u; subtracting
2^15 + z is exact; the product with a bf16 scale is exact; one
round-to-nearest-even to bf16 then gives the oracle's value bit for bit
(signs of zero included, and infinities where the product leaves the bf16
range), for every u in 0..255, zero points across the range and every finite
bf16 scale.  The fp16 path needs no emulation: 1024 + u and 1024 + z are fp16
integers, their difference is exact, and the fp16 multiply rounds once."""

import numpy as np
import torch

from oracle import codecs, quant


def test_byte_placement_reads_two_to_the_15_plus_u():
    u = np.arange(256, dtype=np.uint32)
    x = (np.uint32(0x47000000) | (u << np.uint32(8))).view(np.float32)
    assert np.array_equal(x.astype(np.float64), 32768.0 + u)


def test_fp32_steps_round_once_to_the_oracle_value():
    s_bits = np.arange(1 << 16, dtype=np.uint32)
    s = (s_bits << np.uint32(16)).view(np.float32)
    s = s[np.isfinite(s)]
    u = np.arange(256)
    for z in (0, 1, 77, 128, 200, 255):
        x = (np.uint32(0x47000000) | (u.astype(np.uint32) << np.uint32(8))).view(np.float32)
        d = x - np.float32(32768.0 + z)                       # fp32, exact
        with np.errstate(over="ignore"):
            prod = d[:, None] * s[None, :]                    # fp32 multiply
        got = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy()
        want = quant.dequant_int(np.repeat(u[:, None], s.size, axis=1),
                                 np.repeat(s[None, :].astype(np.float64), 256, axis=0),
                                 np.full((256, s.size), z), 1, "bf16")
        assert np.array_equal(got.view(np.uint16), codecs.dtype_bits("bf16", want)), z
