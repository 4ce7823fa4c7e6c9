"""GPU parity of the W4A8-MXFP4 path against the oracle, through the C ABI:
the repack and the e2m1 -> e4m3 conversion bit for bit, the whole path (per
row FP8 quantization of bf16 activations, block-scaled MMA with the e8m0
weight scales, per-row scale in the epilogue) within |gpu - ref| <= 1e-2 +
1e-2 |ref| per element and relative Frobenius error <= 2e-2."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import DEV, assert_close, to_np
from oracle import codecs, gemm, layout, quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


class MxCase:
    def __init__(self, m, n, k, seed):
        g = synth.rng(seed)
        w = synth.weights_fp32(g, k, n)
        self.x = codecs.bf16(synth.activations_fp32(g, m, k))
        self.codes_kn, self.b_kn = quant.quantize_mxfp4(w)
        self.codes_nk, self.b_nk = quant.pack_mxfp4(self.codes_kn, self.b_kn)
        self.m, self.n, self.k = m, n, k

    def layer(self, **kw):
        from quantized_weight_gemm_run_b300.api import W4A8Linear
        return W4A8Linear(torch.from_numpy(self.codes_nk).to(DEV),
                          torch.from_numpy(self.b_nk).to(DEV), self.n, self.k, **kw)

    def x_dev(self, rows=None):
        x = self.x if rows is None else self.x[:rows]
        return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(DEV)

    def reference(self, rows=None):
        x = self.x if rows is None else self.x[:rows]
        a8, s = gemm.act_quant_fp8(x)
        return gemm.w4a8_reference(a8, s, self.codes_kn, self.b_kn)


def test_mxfp4_repack_and_e4m3_conversion_bit_exact(Q):
    c = MxCase(4, 384, 512, seed=51)
    lin = c.layer()
    torch.cuda.synchronize()
    assert np.array_equal(lin.packed.cpu().numpy(), layout.packed_mxfp4(c.codes_nk, c.b_nk))
    e4 = lin.codes_e4m3().cpu().numpy()
    want = codecs.encode_e4m3(codecs.decode_e2m1(c.codes_kn))
    # e2m1 -0 (code 8) maps to e4m3 -0 (0x80); both sides keep the sign
    assert np.array_equal(e4, want)


def test_all_sixteen_codes_convert(Q):
    # every e2m1 code in every nibble position of a word
    n, k = 128, 128
    codes = np.tile(np.arange(16, dtype=np.uint8), (k * n) // 16).reshape(k, n)
    codes = np.roll(codes, 3, axis=1)
    b = np.full((k // 32, n), 127, dtype=np.uint8)
    cn, bn = quant.pack_mxfp4(codes, b)
    from quantized_weight_gemm_run_b300.api import W4A8Linear
    lin = W4A8Linear(torch.from_numpy(cn).to(DEV), torch.from_numpy(bn).to(DEV), n, k)
    e4 = lin.codes_e4m3().cpu().numpy()
    assert np.array_equal(e4, codecs.encode_e4m3(codecs.decode_e2m1(codes)))


@pytest.mark.parametrize("m,n,k", [(1, 128, 128), (16, 256, 256), (37, 384, 512),
                                   (130, 256, 1024), (300, 640, 384)])
def test_w4a8_small_parity(Q, m, n, k):
    c = MxCase(m, n, k, seed=m + n + k)
    lin = c.layer()
    out = lin(c.x_dev())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), frob=2e-2, what=f"w4a8 {m}x{n}x{k}")


@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("bt", [16, 64, 128])
def test_w4a8_tunings(Q, bt, det):
    c = MxCase(70, 384, 768, seed=9)
    lin = c.layer(tuning=Q.tuning_config(block_tok=bt, max_ctas=11), deterministic=det)
    out = lin(c.x_dev())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), frob=2e-2, what=f"w4a8 bt={bt} det={det}")


def test_w4a8_full_config_all_m(Q):
    s = synth.W4A8_SHAPE
    c = MxCase(max(synth.W4A8_MS), s["n"], s["k"], seed=synth.SEED_W4A8)
    lin = c.layer()
    ref = c.reference()
    for m in synth.W4A8_MS:
        out = lin(c.x_dev(m))
        assert lin.status() == Q.QGEMM_OK
        # per-row quantization makes row r's result independent of the other rows
        assert_close(to_np(out), ref[:m], frob=2e-2, what=f"W4A8 M={m}")


def test_w4a8_rejects_missing_scales(Q):
    c = MxCase(8, 128, 128, seed=3)
    lin = c.layer()
    a8, sc = lin.quantize(c.x_dev())
    out = torch.empty(8, 128, dtype=torch.bfloat16, device=DEV)
    st, need = Q.qgemm_workspace_size(lin.layer, lin.dense, None, 8)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    assert Q.qgemm_run(lin.layer, lin.dense, None, 8, a8, None, lin.packed, None, out,
                       ws, need) == Q.QGEMM_ERR_INVALID_ARG
