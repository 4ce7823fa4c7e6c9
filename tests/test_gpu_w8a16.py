"""GPU parity of W8A16 layers (8-bit integer weights, INT8 symmetric or UINT8
with zero points, scales in the activation dtype) against the oracle, through
the C ABI: the pack and the values fed to the tensor core bit for bit (every
code against every zero point), the GEMM within |gpu - ref| <= 1e-2 +
1e-2 |ref| per element and relative Frobenius error <= 5e-3: dense at small
and full sizes, split-K, grouped and gated; the planner routes these layers
to the tcgen05 kernel at every m."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import DEV, TD, assert_close, to_np
from oracle import codecs, gemm, layout, moe, quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


class W8Case:
    """One W8A16 problem, quantized by the oracle from seeded fp32 data."""

    def __init__(self, m, n, k, g, adt, sym, seed=0, bias=False):
        r = synth.rng(seed)
        w = synth.weights_fp32(r, k, n)
        self.a = codecs.round_dtype(adt)(synth.activations_fp32(r, m, k))
        if sym:
            self.q, self.s = quant.quantize_int_sym(w, g, adt, 8)
            self.z = None
        else:
            self.q, self.s, self.z = quant.quantize_uint_asym(w, g, adt, 8)
        self.m, self.n, self.k, self.g, self.adt, self.sym = m, n, k, g, adt, sym
        self.qweight = quant.pack_int_kn(self.q, 8, sym)
        self.s_bits = codecs.dtype_bits(adt, self.s)
        self.qzeros = None if self.z is None else quant.pack_zeros_bits(self.z, 8)
        self.w_hat = quant.dequant_int(self.q, self.s, self.z, g, adt)
        self.bias = codecs.round_dtype(adt)(r.standard_normal(n) * 0.5) if bias else None

    def layer(self, **kw):
        from quantized_weight_gemm_run_b300.api import W8A16Linear
        bias = None
        if self.bias is not None:
            bias = torch.from_numpy(self.bias.astype(np.float32)).to(TD[self.adt]).to(DEV)
        qz = None if self.qzeros is None else torch.from_numpy(self.qzeros).to(DEV)
        return W8A16Linear(torch.from_numpy(self.qweight).to(DEV),
                           torch.from_numpy(self.s_bits.view(np.int16)).to(DEV), qz,
                           self.n, self.k, self.g, TD[self.adt], bias=bias, **kw)

    def dev_act(self):
        return torch.from_numpy(self.a.astype(np.float32)).to(TD[self.adt]).to(DEV)

    def reference(self):
        return gemm.w4a16_reference(self.a, self.w_hat, self.bias)


@pytest.mark.parametrize("adt,sym,g", [("bf16", True, 128), ("fp16", True, 32),
                                       ("bf16", False, 64), ("fp16", False, 256),
                                       ("bf16", False, 32)])
def test_pack_and_operand_bit_exact(Q, adt, sym, g):
    c = W8Case(8, 384, 512, g, adt, sym, seed=231)
    lin = c.layer()
    torch.cuda.synchronize()
    assert np.array_equal(lin.packed.cpu().numpy(),
                          layout.packed_w8(c.q, c.s_bits, c.z, g, signed=sym))
    deq = lin.dequantized().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, codecs.dtype_bits(adt, c.w_hat))


@pytest.mark.parametrize("adt", ["bf16", "fp16"])
def test_every_code_against_every_zero_point(Q, adt):
    """All 256 x 256 (code, zero point) pairs, under scales of both signs."""
    from quantized_weight_gemm_run_b300.api import W8A16Linear
    k, n, g = 8192, 256, 32
    q = (np.arange(k)[:, None] + np.arange(n)[None, :]) % 256   # every code in every group
    z = np.repeat((np.arange(k // g) % 256)[:, None], n, axis=1)   # one zero point per group
    r = synth.rng(232)
    s = codecs.round_dtype(adt)(r.uniform(0.001, 2.0, (k // g, n)) *
                                np.where(r.random((k // g, n)) < 0.25, -1.0, 1.0))
    lin = W8A16Linear(torch.from_numpy(quant.pack_int_kn(q, 8, False)).to(DEV),
                      torch.from_numpy(codecs.dtype_bits(adt, s).view(np.int16)).to(DEV),
                      torch.from_numpy(quant.pack_zeros_bits(z, 8)).to(DEV), n, k, g, TD[adt])
    deq = lin.dequantized().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, codecs.dtype_bits(adt, quant.dequant_int(q, s, z, g, adt)))


SMALL = [
    # m, n, k, g, adt, sym, bias
    (1, 128, 128, 128, "bf16", True, False),
    (4, 256, 512, 32, "fp16", False, False),
    (16, 384, 1024, 128, "bf16", False, True),
    (37, 384, 512, 64, "fp16", True, False),
    (130, 256, 1024, 128, "bf16", False, True),
    (300, 640, 384, 128, "fp16", True, False),
]


@pytest.mark.parametrize("m,n,k,g,adt,sym,bias", SMALL)
def test_gemm_small_parity(Q, m, n, k, g, adt, sym, bias):
    c = W8Case(m, n, k, g, adt, sym, seed=m + n + k + 11, bias=bias)
    lin = c.layer()
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"w8a16 {m}x{n}x{k} {adt}")


@pytest.mark.parametrize("bt", [16, 32, 64, 128])
@pytest.mark.parametrize("det", [False, True])
def test_split_tiles(Q, bt, det):
    c = W8Case(45, 384, 2048, 128, "bf16", False, seed=233)
    lin = c.layer(tuning=Q.tuning_config(block_tok=bt, max_ctas=7), deterministic=det)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"w8a16 split bt={bt} det={det}")


def test_grouped_ragged_experts(Q):
    from quantized_weight_gemm_run_b300.api import W8A16Linear
    e, n, k, g = 5, 256, 512, 128
    cases = [W8Case(1, n, k, g, "bf16", False, seed=240 + i) for i in range(e)]
    rows = [7, 0, 40, 1, 19]
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    a = codecs.bf16(synth.activations_fp32(synth.rng(241), int(offsets[-1]), k))
    for bt in (16, 64):
        lin = W8A16Linear(torch.from_numpy(np.concatenate([c.qweight for c in cases])).to(DEV),
                          torch.from_numpy(np.concatenate([c.s_bits for c in cases])
                                           .view(np.int16)).to(DEV),
                          torch.from_numpy(np.concatenate([c.qzeros for c in cases])).to(DEV),
                          n, k, g, torch.bfloat16, num_experts=e,
                          tuning=Q.tuning_config(block_tok=bt))
        out = lin.run_grouped(torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(DEV),
                              torch.from_numpy(offsets).to(DEV))
        assert lin.status() == Q.QGEMM_OK
        got = to_np(out)
        for i in range(e):
            r0, r1 = offsets[i], offsets[i + 1]
            if r1 > r0:
                assert_close(got[r0:r1], a[r0:r1] @ cases[i].w_hat, what=f"bt={bt} expert {i}")


def test_gated(Q):
    c = W8Case(37, 384, 512, 128, "bf16", True, seed=242)
    lin = c.layer(gated=True)
    torch.cuda.synchronize()
    il = layout.glu_interleave_columns
    assert np.array_equal(lin.packed.cpu().numpy(),
                          layout.packed_w8(il(c.q), il(c.s_bits), None, 128, signed=True))
    deq = lin.dequantized().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, codecs.dtype_bits("bf16", c.w_hat))
    out = lin(c.dev_act())
    assert out.shape == (37, 192) and lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), moe.silu_mul(codecs.bf16(c.reference()), 192), what="w8a16 gated")


@pytest.mark.parametrize("m,adt", [(16, "fp16"), (256, "bf16")])
def test_full_size_4096(Q, m, adt):
    """Every element of M x 4096 x 4096 against the oracle."""
    c = W8Case(m, 4096, 4096, 128, adt, adt == "fp16", seed=243 + m)
    lin = c.layer()
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"w8a16 {m}x4096x4096 {adt}")


def test_plan_and_rejections(Q):
    c = W8Case(8, 256, 256, 128, "bf16", False, seed=244)
    lin = c.layer()
    st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, 8)
    assert st == Q.QGEMM_OK
    assert "kernel=w4a16_tcgen05_swapab" in rec and "weights=uint8_zp" in rec
    forced = c.layer(tuning=Q.tuning_config(kernel=2))
    with pytest.raises(Q.QGemmError):
        forced(c.dev_act())
    # zero points are required for UINT8
    packed = torch.empty_like(lin.packed)
    assert Q.qgemm_pack_weights(lin.layer, torch.from_numpy(c.qweight).to(DEV),
                                torch.from_numpy(c.s_bits.view(np.int16)).to(DEV), None,
                                packed) == Q.QGEMM_ERR_INVALID_ARG
