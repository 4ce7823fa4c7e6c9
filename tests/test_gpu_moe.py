"""GPU parity of the grouped-MoE path and the FP8 activation quantizer against
the oracle, through the C ABI: the permutation and the FP8 codes bit for bit;
the SiLU gate and the combine within one bf16 unit in the last place (fp32
library exp and fp32 sums against float64); the grouped GEMMs and the whole
layer within the acceptance tolerance."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import DEV, assert_close, to_np
from oracle import codecs, gemm, moe, quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


def _bf16_dev(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(DEV)


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16).astype(np.int64)


def _ulp_diff_bf16(a_bits, b_bits):
    def ordered(b):
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def _permute(Q, ids, e, a):
    t, topk = ids.shape
    hidden = a.shape[1]
    offs = torch.empty(e + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(t * topk, dtype=torch.int32, device=DEV)
    inv = torch.empty(t * topk, dtype=torch.int32, device=DEV)
    a_perm = torch.empty(t * topk, hidden, dtype=torch.bfloat16, device=DEV)
    Q.check(Q.qgemm_moe_permute(torch.from_numpy(ids).to(DEV), t, topk, e, offs, perm, inv,
                                _bf16_dev(a), a_perm, hidden))
    torch.cuda.synchronize()
    return offs.cpu().numpy(), perm.cpu().numpy(), inv.cpu().numpy(), a_perm


@pytest.mark.parametrize("t,topk,e", [(37, 3, 6), (1, 8, 64), (4096, 8, 64), (3000, 2, 256),
                                      (2048, 8, 4)])
def test_permute_bit_exact(Q, t, topk, e):
    g = np.random.default_rng(t + e)
    ids = g.integers(0, max(1, e - 1), (t, topk)).astype(np.int32)   # the last expert gets none
    a = codecs.bf16(g.standard_normal((t, 64)))
    offs, perm, inv, a_perm = _permute(Q, ids, e, a)
    o_ref, p_ref = moe.permute(ids, e)
    assert np.array_equal(offs, o_ref)
    assert np.array_equal(perm, p_ref)
    assert np.array_equal(perm[inv], np.arange(t * topk))
    assert np.array_equal(to_np(a_perm), moe.gather_rows(a, p_ref, topk))


def test_permute_out_of_range_ids_stay_memory_safe(Q):
    ids = np.array([[0, 5], [-1, 2], [2, 99]], dtype=np.int32)
    a = codecs.bf16(np.arange(3 * 8, dtype=np.float64).reshape(3, 8))
    offs, perm, inv, _ = _permute(Q, ids, 6, a)
    assert offs[-1] == 4                              # four valid slots
    assert sorted(perm.tolist()) == list(range(6))    # still a permutation
    assert set(perm[4:].tolist()) == {2, 5}           # invalid slots after the last expert


def test_silu_mul_within_one_ulp(Q):
    g = np.random.default_rng(3)
    rows, inter = 300, 1408
    gu = codecs.bf16(g.standard_normal((rows, 2 * inter)) * 2.0)
    h = torch.empty(rows, inter, dtype=torch.bfloat16, device=DEV)
    Q.check(Q.qgemm_moe_silu_mul(_bf16_dev(gu), rows, inter, h))
    ref = moe.silu_mul(gu, inter)
    d = _ulp_diff_bf16(_bits(h), codecs.bf16_bits(ref).astype(np.int64))
    assert d.max() <= 1 and (d > 0).mean() < 0.01


def test_combine_within_one_ulp(Q):
    g = np.random.default_rng(4)
    t, topk, hidden = 77, 8, 2048
    ids = np.stack([g.permutation(16)[:topk] for _ in range(t)]).astype(np.int32)
    wts = g.uniform(0, 0.3, (t, topk)).astype(np.float32)
    _, perm = moe.permute(ids, 16)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    y2 = codecs.bf16(g.standard_normal((t * topk, hidden)))
    y = torch.empty(t, hidden, dtype=torch.bfloat16, device=DEV)
    Q.check(Q.qgemm_moe_combine(_bf16_dev(y2), torch.from_numpy(inv).to(DEV),
                                torch.from_numpy(wts).to(DEV), t, topk, hidden, y))
    ref = moe.combine(y2, perm, wts, topk)
    d = _ulp_diff_bf16(_bits(y), codecs.bf16_bits(ref).astype(np.int64))
    assert d.max() <= 1


@pytest.mark.parametrize("m", synth.W4A8_MS + [3])
def test_act_quant_fp8_bit_exact(Q, m):
    g = synth.rng(synth.SEED_W4A8)
    k = synth.W4A8_SHAPE["k"]
    x = codecs.bf16(synth.activations_fp32(g, m, k))
    if m >= 3:
        x[1] = 0.0                                   # all-zero row: scale 1, codes 0
        x[2, :5] = [3e4, -3e4, 1e-30, -0.0, 448.0]   # wide dynamic range in one row
        x = codecs.bf16(x)
    a8 = torch.empty(m, k, dtype=torch.uint8, device=DEV)
    sc = torch.empty(m, dtype=torch.float32, device=DEV)
    Q.check(Q.qgemm_quantize_act_fp8(_bf16_dev(x), m, k, a8, sc))
    codes, s = gemm.act_quant_fp8(x)
    assert np.array_equal(sc.cpu().numpy(), s)
    assert np.array_equal(a8.cpu().numpy(), codes)


# ------------------------------------------------------------------ the layer

class MoEWeights:
    """The grouped-MoE workload's experts, quantized by the oracle."""

    def __init__(self, e, hidden, inter, gsz, seed):
        g = synth.rng(seed)
        self.e, self.hidden, self.inter, self.g = e, hidden, inter, gsz
        self.q1, self.s1, self.q2, self.s2 = [], [], [], []
        for _ in range(e):
            q, s = quant.quantize_int4_sym(synth.weights_fp32(g, hidden, 2 * inter), gsz, "bf16")
            self.q1.append(q.astype(np.int8))
            self.s1.append(s)
        for _ in range(e):
            q, s = quant.quantize_int4_sym(synth.weights_fp32(g, inter, hidden), gsz, "bf16")
            self.q2.append(q.astype(np.int8))
            self.s2.append(s)
        self.gen = g
        self._c1, self._c2 = {}, {}

    def w1_hat(self, i):
        if i not in self._c1:
            self._c1[i] = quant.dequant_int(self.q1[i], self.s1[i], None, self.g, "bf16")
        return self._c1[i]

    def w2_hat(self, i):
        if i not in self._c2:
            self._c2[i] = quant.dequant_int(self.q2[i], self.s2[i], None, self.g, "bf16")
        return self._c2[i]

    def layer(self, topk, gated=True):
        from quantized_weight_gemm_run_b300.api import MoELayer, W4A16Linear

        def stack(qs, ss):
            qw = np.concatenate([quant.pack_int4_kn(q, True) for q in qs])
            sc = np.concatenate([codecs.bf16_bits(s) for s in ss]).view(np.int16)
            return torch.from_numpy(qw).to(DEV), torch.from_numpy(sc).to(DEV)

        l1 = W4A16Linear(*stack(self.q1, self.s1), None, 2 * self.inter, self.hidden, self.g,
                         torch.bfloat16, num_experts=self.e, gated=gated)
        l2 = W4A16Linear(*stack(self.q2, self.s2), None, self.hidden, self.inter, self.g,
                         torch.bfloat16, num_experts=self.e)
        return MoELayer(l1, l2, self.e, topk), l1, l2


@pytest.fixture(scope="module")
def moe_full():
    s = synth.MOE_SHAPE
    w = MoEWeights(s["experts"], s["hidden"], s["inter"], s["group"], synth.SEED_MOE)
    return w


def test_moe_layer_small_all_stages(Q):
    w = MoEWeights(8, 256, 128, 128, seed=17)
    layer, l1, l2 = w.layer(3, gated=False)   # the unfused path keeps GU for the check
    g = synth.rng(18)
    t = 45
    x = codecs.bf16(synth.activations_fp32(g, t, 256))
    ids, wts = moe.route(synth.router_logits_fp32(g, t, 8), 3)
    y, b = layer(_bf16_dev(x), torch.from_numpy(ids).to(DEV), torch.from_numpy(wts).to(DEV),
                 keep=True)
    assert l1.status() == Q.QGEMM_OK and l2.status() == Q.QGEMM_OK
    ref = moe.moe_layer(x, ids, wts, w.w1_hat, w.w2_hat, 8, 128)
    r = t * 3
    assert np.array_equal(b["offsets"].cpu().numpy(), ref["offsets"])
    # each stage against the oracle applied to the GPU's own previous stage
    gu = to_np(b["gu"][:r])
    assert_close(gu, moe.grouped_gemm(to_np(b["a_perm"][:r]), ref["offsets"], w.w1_hat, "bf16"),
                 what="GEMM1")
    h = to_np(b["h"][:r])
    d = _ulp_diff_bf16(_bits(b["h"][:r]), codecs.bf16_bits(moe.silu_mul(gu, 128)).astype(np.int64))
    assert d.max() <= 1
    assert_close(to_np(b["y2"][:r]), moe.grouped_gemm(h, ref["offsets"], w.w2_hat, "bf16"),
                 what="GEMM2")
    assert_close(to_np(y), ref["y"], what="layer")


@pytest.mark.parametrize("gated", [True, False])
@pytest.mark.parametrize("t", [16, 256])
def test_moe_layer_full_config(Q, moe_full, t, gated):
    s = synth.MOE_SHAPE
    layer, l1, l2 = moe_full.layer(s["topk"], gated=gated)
    g = synth.rng(synth.SEED_MOE + t)
    x = codecs.bf16(synth.activations_fp32(g, t, s["hidden"]))
    ids, wts = moe.route(synth.router_logits_fp32(g, t, s["experts"]), s["topk"])
    y = layer(_bf16_dev(x), torch.from_numpy(ids).to(DEV), torch.from_numpy(wts).to(DEV))
    assert l1.status() == Q.QGEMM_OK and l2.status() == Q.QGEMM_OK
    ref = moe.moe_layer(x, ids, wts, moe_full.w1_hat, moe_full.w2_hat, s["experts"], s["inter"])
    assert_close(to_np(y), ref["y"], what=f"MoE T={t}")


def test_moe_layer_t4096_every_token(Q, moe_full):
    """T = 4096 (32768 permuted rows, 128-row expert tiles across ragged expert
    boundaries): every token of the layer's output against the oracle."""
    s = synth.MOE_SHAPE
    t, topk = 4096, s["topk"]
    layer, l1, l2 = moe_full.layer(topk)
    g = synth.rng(synth.SEED_MOE + t)
    x = codecs.bf16(synth.activations_fp32(g, t, s["hidden"]))
    ids, wts = moe.route(synth.router_logits_fp32(g, t, s["experts"]), topk)
    y = layer(_bf16_dev(x), torch.from_numpy(ids).to(DEV), torch.from_numpy(wts).to(DEV))
    assert l1.status() == Q.QGEMM_OK and l2.status() == Q.QGEMM_OK
    ref = moe.moe_layer(x, ids, wts, moe_full.w1_hat, moe_full.w2_hat, s["experts"],
                        s["inter"])["y"]
    assert_close(to_np(y), ref, what="MoE T=4096 every token")
