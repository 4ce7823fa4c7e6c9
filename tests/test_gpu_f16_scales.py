"""GPU parity of W4A16 layers with fp16 scales against bf16 activations,
through the C ABI: each weight is (q - z) * s rounded once to bf16, the scale
not rounded to bf16 first.  The pack and the values fed to the tensor core
bit for bit (every code and zero point under every finite scale), the GEMM within
|gpu - ref| <= 1e-2 + 1e-2 |ref| per element and relative Frobenius error
<= 5e-3: dense at small and full sizes, split-K, grouped and gated; the
planner routes dense layers of at most 16 rows to the small-M kernel, which
must feed the MMA the same operand bits, and the rest to the tcgen05 kernel."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import DEV, Case, assert_close, linear, to_np
from oracle import codecs, layout, moe, quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


def _case(m, n, k, g, sym, seed, bias=False):
    return Case(m, n, k, g, "bf16", sym, seed=seed, bias=bias, sdt="fp16")


@pytest.mark.parametrize("sym,g", [(True, 128), (False, 32), (False, 64), (True, 256)])
def test_pack_and_operand_bit_exact(Q, sym, g):
    c = _case(8, 384, 512, g, sym, seed=131)
    lin = linear(c)
    torch.cuda.synchronize()
    assert np.array_equal(lin.packed.cpu().numpy(),
                          layout.packed_w4(c.q, c.s_bits, c.z, g, signed=sym))
    deq = lin.dequantized().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, codecs.dtype_bits("bf16", c.w_hat))
    # the scales are used unrounded: some weights differ from bf16-rounded scales'
    pre = quant.dequant_int(c.q, codecs.round_dtype("bf16")(c.s), c.z, g, "bf16")
    assert np.any(pre != c.w_hat)


def test_every_code_zero_and_scale(Q):
    """Every UINT4 code against every zero point, under every finite fp16
    scale of either sign (subnormals included)."""
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    k, n, g = 4096, 512, 32
    q = (np.arange(k)[:, None] + np.arange(n)[None, :]) % 16   # every code in every group
    z = np.repeat((np.arange(k // g) % 16)[:, None], n, axis=1)   # one zero point per group
    finite = np.concatenate([np.arange(0x7C00), 0x8000 + np.arange(0x7C00)]).astype(np.uint16)
    bits = np.resize(np.random.default_rng(7).permutation(finite), (k // g) * n)
    s = bits.view(np.float16).astype(np.float64).reshape(k // g, n)
    lin = W4A16Linear(torch.from_numpy(quant.pack_int4_kn(q, False)).to(DEV),
                      torch.from_numpy(bits.view(np.int16).reshape(k // g, n)).to(DEV),
                      torch.from_numpy(quant.pack_zeros(z)).to(DEV), n, k, g, torch.bfloat16,
                      scale_dtype=torch.float16)
    deq = lin.dequantized().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, codecs.dtype_bits("bf16", quant.dequant_int(q, s, z, g, "bf16")))


SMALL = [
    # m, n, k, g, sym, bias
    (1, 128, 128, 128, True, False),
    (8, 256, 512, 32, False, False),
    (16, 384, 1024, 128, False, True),
    (37, 384, 512, 64, True, False),
    (130, 256, 1024, 128, False, True),
    (300, 640, 384, 128, True, False),
]


@pytest.mark.parametrize("m,n,k,g,sym,bias", SMALL)
def test_gemm_small_parity(Q, m, n, k, g, sym, bias):
    c = _case(m, n, k, g, sym, seed=m + n + k + 7, bias=bias)
    lin = linear(c)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"f16 scales {m}x{n}x{k}")


@pytest.mark.parametrize("bt", [16, 128])
@pytest.mark.parametrize("det", [False, True])
def test_split_tiles(Q, bt, det):
    c = _case(45, 384, 2048, 128, False, seed=133)
    lin = linear(c, tuning=Q.tuning_config(block_tok=bt, max_ctas=7), deterministic=det)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"f16 scales split bt={bt} det={det}")


def test_grouped_ragged_experts(Q):
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    e, n, k, g = 5, 256, 512, 128
    cases = [_case(1, n, k, g, False, seed=140 + i) for i in range(e)]
    rows = [7, 0, 40, 1, 19]
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    a = codecs.bf16(synth.activations_fp32(synth.rng(141), int(offsets[-1]), k))
    lin = W4A16Linear(torch.from_numpy(np.concatenate([c.qweight for c in cases])).to(DEV),
                      torch.from_numpy(np.concatenate([c.s_bits for c in cases])
                                       .view(np.int16)).to(DEV),
                      torch.from_numpy(np.concatenate([c.qzeros for c in cases])).to(DEV),
                      n, k, g, torch.bfloat16, num_experts=e, scale_dtype=torch.float16)
    out = lin.run_grouped(torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(DEV),
                          torch.from_numpy(offsets).to(DEV))
    assert lin.status() == Q.QGEMM_OK
    got = to_np(out)
    for i in range(e):
        r0, r1 = offsets[i], offsets[i + 1]
        if r1 > r0:
            assert_close(got[r0:r1], a[r0:r1] @ cases[i].w_hat, what=f"expert {i}")


def test_gated(Q):
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    c = _case(37, 384, 512, 128, True, seed=142)
    qw, sc, qz = c.dev_weights()
    lin = W4A16Linear(qw, sc, qz, c.n, c.k, c.g, torch.bfloat16, gated=True,
                      scale_dtype=torch.float16)
    out = lin(c.dev_act())
    assert out.shape == (37, 192) and lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), moe.silu_mul(codecs.bf16(c.reference()), 192), what="gated")


def test_full_size_m16_and_m256(Q):
    """Every element of M = 16 and M = 256 over N = K = 4096 against the oracle."""
    for m in (16, 256):
        c = _case(m, 4096, 4096, 128, False, seed=143 + m)
        lin = linear(c)
        out = lin(c.dev_act())
        assert lin.status() == Q.QGEMM_OK
        assert_close(to_np(out), c.reference(), what=f"f16 scales {m}x4096x4096")


def test_plan_takes_small_m_kernel_up_to_16_rows(Q):
    c = _case(8, 256, 256, 128, True, seed=144)
    lin = linear(c)
    for m, kern in ((8, "w4a16_mma_sync_smallm"), (16, "w4a16_mma_sync_smallm"),
                    (17, "w4a16_tcgen05_swapab")):
        st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, m)
        assert st == Q.QGEMM_OK
        assert f"kernel={kern}" in rec and "scales=fp16 act=bf16" in rec, rec
    # forced onto either kernel, the two agree within the GEMM tolerance
    x = c.dev_act()
    small = linear(c, tuning=Q.tuning_config(kernel=2))(x)
    big = linear(c, tuning=Q.tuning_config(kernel=1))(x)
    assert_close(to_np(small), c.reference(), what="f16 scales small-M kernel")
    assert_close(to_np(big), c.reference(), what="f16 scales tcgen05 kernel")


def test_small_m_kernel_operands_every_code_zero_and_scale(Q):
    """The small-M kernel's own dequant of fp16 scales against bf16
    activations: one-hot activation rows pick single weight rows, so each
    output is one dequantized weight (the product with 1.0 and the fp32 sums
    of zeros are exact).  Eight calls of 16 rows take one row of every group:
    every code against every zero point under every finite fp16 scale of
    either sign, compared with the oracle's bf16((q - z) s) (+0 and -0 equal)."""
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    k, n, g = 4096, 512, 32
    q = (np.arange(k)[:, None] + np.arange(n)[None, :]) % 16
    z = np.repeat((np.arange(k // g) % 16)[:, None], n, axis=1)
    finite = np.concatenate([np.arange(0x7C00), 0x8000 + np.arange(0x7C00)]).astype(np.uint16)
    bits = np.resize(np.random.default_rng(9).permutation(finite), (k // g) * n)
    s = bits.view(np.float16).astype(np.float64).reshape(k // g, n)
    lin = W4A16Linear(torch.from_numpy(quant.pack_int4_kn(q, False)).to(DEV),
                      torch.from_numpy(bits.view(np.int16).reshape(k // g, n)).to(DEV),
                      torch.from_numpy(quant.pack_zeros(z)).to(DEV), n, k, g, torch.bfloat16,
                      scale_dtype=torch.float16, tuning=Q.tuning_config(kernel=2))
    w_hat = quant.dequant_int(q, s, z, g, "bf16")
    groups = k // g
    for call in range(groups // 16):
        rows = [(call * 16 + i) * g + (call * 7 + i) % g for i in range(16)]
        x = np.zeros((16, k), dtype=np.float32)
        x[np.arange(16), rows] = 1.0
        out = lin(torch.from_numpy(x).to(torch.bfloat16).to(DEV))
        assert lin.status() == Q.QGEMM_OK
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.array_equal(got, w_hat[rows]), f"call {call}"
