"""GPU parity of W3A16 layers (GPTQ INT3 weights, or UINT3 with zero points;
each column's 3-bit codes a bit stream along K) against the oracle, through
the C ABI: the pack bit for bit against the oracle's layout reading (the
codes in the 4-bit blocks), the values fed to the tensor core bit for bit,
and the GEMM within |gpu - ref| <= 1e-2 + 1e-2 |ref| per element and
relative Frobenius error <= 5e-3, on the small-M and the tcgen05 kernels,
split tiles, fp16 scales with bf16 activations, grouped and gated layers,
and the sweep's full shapes."""

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


class W3Case:
    """One W3A16 problem, quantized by the oracle from seeded fp32 data."""

    def __init__(self, m, n, k, g, adt, sym, seed=0, bias=False, sdt=None):
        r = synth.rng(seed)
        w = synth.weights_fp32(r, k, n)
        sdt = adt if sdt is None else sdt
        self.a = codecs.round_dtype(adt)(synth.activations_fp32(r, m, k))
        if sym:
            self.q, self.s = quant.quantize_int_sym(w, g, sdt, 3)
            self.z = None
        else:
            self.q, self.s, self.z = quant.quantize_uint_asym(w, g, sdt, 3)
        self.m, self.n, self.k, self.g, self.adt, self.sym, self.sdt = m, n, k, g, adt, sym, sdt
        self.qweight = quant.pack_int_kn(self.q, 3, sym)
        self.s_bits = codecs.dtype_bits(sdt, self.s)
        self.qzeros = None if self.z is None else quant.pack_zeros_bits(self.z, 3)
        self.w_hat = quant.dequant_int(self.q, self.s, self.z, g, adt)
        self.bias = codecs.round_dtype(adt)(r.standard_normal(n) * 0.5) if bias else None

    def layer(self, **kw):
        from quantized_weight_gemm_run_b300.api import W3A16Linear
        bias = None
        if self.bias is not None:
            bias = torch.from_numpy(self.bias.astype(np.float32)).to(TD[self.adt]).to(DEV)
        qz = None if self.qzeros is None else torch.from_numpy(self.qzeros).to(DEV)
        return W3A16Linear(torch.from_numpy(self.qweight).to(DEV),
                           torch.from_numpy(self.s_bits.view(np.int16)).to(DEV), qz,
                           self.n, self.k, self.g, TD[self.adt], bias=bias,
                           scale_dtype=TD[self.sdt], **kw)

    def dev_act(self):
        return torch.from_numpy(self.a.astype(np.float32)).to(TD[self.adt]).to(DEV)

    def reference(self):
        return gemm.w4a16_reference(self.a, self.w_hat, self.bias)


@pytest.mark.parametrize("adt,sym,g", [("bf16", True, 128), ("fp16", True, 32),
                                       ("bf16", False, 64), ("fp16", False, 256)])
def test_pack_and_operand_bit_exact(Q, adt, sym, g):
    c = W3Case(8, 384, 512, g, adt, sym, seed=331)
    lin = c.layer()
    torch.cuda.synchronize()
    assert np.array_equal(lin.packed.cpu().numpy(),
                          layout.packed_w3(c.q, c.s_bits, c.z, g, signed=sym))
    deq = lin.dequantized().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, codecs.dtype_bits(adt, c.w_hat))


@pytest.mark.parametrize("adt", ["bf16", "fp16"])
def test_every_code_against_every_zero_point(Q, adt):
    """All 8 x 8 (code, zero point) pairs, under scales of both signs."""
    from quantized_weight_gemm_run_b300.api import W3A16Linear
    k, n, g = 2048, 256, 32
    q = (np.arange(k)[:, None] + np.arange(n)[None, :]) % 8
    z = np.repeat((np.arange(k // g) % 8)[:, None], n, axis=1)
    r = synth.rng(332)
    s = codecs.round_dtype(adt)(r.uniform(0.001, 2.0, (k // g, n)) *
                                np.where(r.random((k // g, n)) < 0.25, -1.0, 1.0))
    lin = W3A16Linear(torch.from_numpy(quant.pack_int_kn(q, 3, False)).to(DEV),
                      torch.from_numpy(codecs.dtype_bits(adt, s).view(np.int16)).to(DEV),
                      torch.from_numpy(quant.pack_zeros_bits(z, 3)).to(DEV), n, k, g, TD[adt])
    deq = lin.dequantized().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, codecs.dtype_bits(adt, quant.dequant_int(q, s, z, g, adt)))


SMALL = [
    # m, n, k, g, adt, sym, bias, sdt
    (1, 128, 128, 128, "bf16", True, False, None),
    (4, 256, 512, 32, "fp16", False, False, None),
    (16, 384, 1024, 128, "bf16", False, True, None),
    (37, 384, 512, 64, "fp16", True, False, None),
    (130, 256, 1024, 128, "bf16", False, True, "fp16"),   # fp16 scales, bf16 activations
    (300, 640, 384, 128, "fp16", True, False, None),
]


@pytest.mark.parametrize("m,n,k,g,adt,sym,bias,sdt", SMALL)
def test_gemm_small_parity(Q, m, n, k, g, adt, sym, bias, sdt):
    c = W3Case(m, n, k, g, adt, sym, seed=m + n + k + 13, bias=bias, sdt=sdt)
    lin = c.layer()
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"w3a16 {m}x{n}x{k} {adt}")


@pytest.mark.parametrize("kernel", [1, 2])
def test_both_kernels_at_small_m(Q, kernel):
    c = W3Case(9, 512, 2048, 128, "bf16", False, seed=334)
    lin = c.layer(tuning=Q.tuning_config(kernel=kernel))
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"w3a16 kernel {kernel}")


@pytest.mark.parametrize("bt", [16, 64, 128])
@pytest.mark.parametrize("det", [False, True])
def test_split_tiles(Q, bt, det):
    c = W3Case(45, 384, 2048, 128, "bf16", True, seed=335)
    lin = c.layer(tuning=Q.tuning_config(block_tok=bt, max_ctas=7), deterministic=det)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"w3a16 split bt={bt} det={det}")


def test_grouped_gated_layer(Q):
    """A small MoE layer with 3-bit experts: the gated gate|up GEMM and the
    down GEMM over router-permuted rows, against the oracle's layer."""
    from quantized_weight_gemm_run_b300.api import MoELayer, W3A16Linear
    e, topk, hid, inter, t, g = 6, 2, 256, 128, 29, 128
    r = synth.rng(336)
    w1 = synth.expert_weights_fp32(r, e, hid, 2 * inter)
    w2 = synth.expert_weights_fp32(r, e, inter, hid)
    x = codecs.bf16(synth.activations_fp32(r, t, hid))
    ids, wts = moe.route(synth.router_logits_fp32(r, t, e), topk)
    q1 = [quant.quantize_int_sym(w1[i], g, "bf16", 3) for i in range(e)]
    q2 = [quant.quantize_int_sym(w2[i], g, "bf16", 3) for i in range(e)]

    def stack(qs):
        qw = np.concatenate([quant.pack_int_kn(qq, 3, True) for qq, _ in qs])
        sc = np.concatenate([codecs.bf16_bits(ss) for _, ss in qs]).view(np.int16)
        return torch.from_numpy(qw).to(DEV), torch.from_numpy(sc).to(DEV)
    l1 = W3A16Linear(*stack(q1), None, 2 * inter, hid, g, torch.bfloat16, num_experts=e,
                     gated=True)
    l2 = W3A16Linear(*stack(q2), None, hid, inter, g, torch.bfloat16, num_experts=e)
    y = MoELayer(l1, l2, e, topk)(torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
                                  .to(DEV), torch.from_numpy(ids).to(DEV),
                                  torch.from_numpy(wts).to(DEV))
    assert l1.status() == Q.QGEMM_OK and l2.status() == Q.QGEMM_OK
    w1h = [quant.dequant_int(qq, ss, None, g, "bf16") for qq, ss in q1]
    w2h = [quant.dequant_int(qq, ss, None, g, "bf16") for qq, ss in q2]
    ref = moe.moe_layer(x, ids, wts, lambda i: w1h[i], lambda i: w2h[i], e, inter)["y"]
    assert_close(to_np(y), ref, what="w3a16 MoE layer")


@pytest.mark.parametrize("n,k", synth.W4A16_ASYM_SHAPES)
def test_full_size_sweep_shapes(Q, n, k):
    c = W3Case(1024, n, k, 128, "bf16", False, seed=synth.SEED_W4A16_ASYM + 30)
    lin = c.layer()
    x = c.dev_act()
    ref = c.reference()
    for m in (1, 16, 1024):
        out = lin(x[:m].contiguous())
        assert lin.status() == Q.QGEMM_OK
        assert_close(to_np(out), ref[:m], what=f"w3a16 M={m} N={n} K={k}")


def test_rejections(Q):
    # UINT3 needs uint3 zero points; INT3 takes none
    bad = Q.layer_config(256, 256, 128, Q.QGEMM_W_UINT3_ZP, Q.QGEMM_S_BF16, Q.QGEMM_Z_UINT4,
                         Q.QGEMM_BF16, Q.QGEMM_BF16)
    st, _ = Q.qgemm_packed_size(bad)
    assert st == Q.QGEMM_ERR_UNSUPPORTED
    bad = Q.layer_config(256, 256, 128, Q.QGEMM_W_INT3_SYM, Q.QGEMM_S_BF16, Q.QGEMM_Z_UINT3,
                         Q.QGEMM_BF16, Q.QGEMM_BF16)
    st, _ = Q.qgemm_packed_size(bad)
    assert st == Q.QGEMM_ERR_UNSUPPORTED
