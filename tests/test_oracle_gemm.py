"""Pins for the GEMM references, the FP8 activation quantizer and the MoE
layer: brute force on tiny problems, exact special cases, invariants."""

import math

import numpy as np
import pytest

import synth
from oracle import codecs, gemm, moe, quant


def _brute_gemm(a, w, bias=None):
    m, k = a.shape
    n = w.shape[1]
    out = [[0.0] * n for _ in range(m)]
    for i in range(m):
        for j in range(n):
            acc = math.fsum(float(a[i, kk]) * float(w[kk, j]) for kk in range(k))
            out[i][j] = acc + (0.0 if bias is None else float(bias[j]))
    return np.array(out)


@pytest.mark.parametrize("adt,signed", [("fp16", True), ("bf16", False)])
def test_w4a16_brute_force_4x8x32(adt, signed):
    g = synth.rng(20)
    w = synth.weights_fp32(g, 32, 8)
    a = codecs.round_dtype(adt)(synth.activations_fp32(g, 4, 32))
    bias = codecs.round_dtype(adt)(g.standard_normal(8) * 0.1)
    if signed:
        q, s = quant.quantize_int4_sym(w, 32, adt)
        z = None
    else:
        q, s, z = quant.quantize_uint4_asym(w, 32, adt)
    # standard format round trip, then the oracle path
    qw = quant.pack_int4_kn(q, signed)
    qz = None if z is None else quant.pack_zeros(z)
    w_hat = gemm.dense_from_standard_int(qw, codecs.dtype_bits(adt, s), qz, 32, 32, adt, adt, signed)
    # brute-force dequant from the definition, element by element
    wb = np.zeros((32, 8))
    for kk in range(32):
        for n in range(8):
            zz = 0 if z is None else z[kk // 32, n]
            wb[kk, n] = float(codecs.round_dtype(adt)((q[kk, n] - zz) * s[kk // 32, n]))
    assert np.array_equal(w_hat, wb)
    ref = gemm.w4a16_reference(a, w_hat, bias)
    brute = _brute_gemm(a, wb, bias)
    assert np.allclose(ref, brute, rtol=1e-13, atol=1e-14)
    out = gemm.w4a16_output(a, w_hat, adt, bias)
    assert np.array_equal(out, codecs.round_dtype(adt)(brute))


def test_w4a16_unit_scale_reduces_to_integer_matmul():
    g = np.random.default_rng(21)
    q = g.integers(-8, 8, (256, 16))
    a_int = g.integers(-50, 50, (8, 256))
    w_hat = quant.dequant_int(q, np.ones((2, 16)), None, 128, "bf16")
    ref = gemm.w4a16_reference(a_int.astype(np.float64), w_hat)
    assert np.array_equal(ref, (a_int @ q).astype(np.float64))


def test_w4a16_transposed_operands_detected():
    # a wrong orientation (W^T or A^T) changes the result of a non-square case
    g = synth.rng(22)
    a = codecs.bf16(synth.activations_fp32(g, 3, 32))
    w = codecs.bf16(synth.weights_fp32(g, 32, 32))
    ref = gemm.w4a16_reference(a, w)
    assert not np.allclose(ref, a @ w.T)


def test_act_quant_fp8_properties_and_brute_force():
    g = synth.rng(23)
    x = codecs.bf16(synth.activations_fp32(g, 6, 64))
    x[3] = 0.0
    codes, s = gemm.act_quant_fp8(x)
    assert s.dtype == np.float32 and s[3] == 1.0 and np.all(codes[3] == 0)
    for m in range(6):
        amax = np.float32(np.max(np.abs(x[m].astype(np.float32))))
        sm = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))
        assert s[m] == sm
        for k in range(64):
            v = np.float32(np.float32(x[m, k]) / sm)
            assert codes[m, k] == codecs.encode_e4m3(float(v))
        if amax > 0:
            top = np.argmax(np.abs(x[m]))
            assert codecs.decode_e4m3(codes[m, top]) in (448.0, -448.0)


def test_w4a8_brute_force_and_unit_scale_case():
    g = synth.rng(24)
    w = synth.weights_fp32(g, 64, 8)
    x = codecs.bf16(synth.activations_fp32(g, 4, 64))
    codes, b = quant.quantize_mxfp4(w)
    a8, s = gemm.act_quant_fp8(x)
    ref = gemm.w4a8_reference(a8, s, codes, b)
    brute = np.zeros((4, 8))
    for m in range(4):
        for n in range(8):
            tot = 0.0
            for kk in range(64):
                tot += (float(codecs.decode_e4m3(a8[m, kk])) * float(codecs.decode_e2m1(codes[kk, n]))
                        * 2.0 ** (int(b[kk // 32, n]) - 127))
            brute[m, n] = tot * float(s[m])
    assert np.allclose(ref, brute, rtol=1e-12, atol=1e-15)
    # unit scales: the plain product of decoded e4m3 and e2m1 values
    bu = np.full_like(b, 127)
    ref1 = gemm.w4a8_reference(a8, np.ones(4, dtype=np.float32), codes, bu)
    assert np.array_equal(ref1, codecs.decode_e4m3(a8) @ codecs.decode_e2m1(codes))


def test_check_close_flags_a_planted_error():
    ref = np.linspace(-2, 2, 100).reshape(10, 10)
    ok, _, _ = gemm.check_close(ref + 1e-4, ref)
    assert ok
    bad = ref.copy()
    bad[3, 3] += 0.2
    ok, worst, _ = gemm.check_close(bad, ref)
    assert not ok and worst > 0


# ------------------------------------------------------------------ MoE


def test_route_ties_and_topk():
    logits = np.zeros((2, 6), dtype=np.float32)
    logits[0, [1, 4]] = 1.0            # tie between experts 1 and 4, then all zero
    logits[1] = [0, 5, 3, 5, 1, 2]
    ids, w = moe.route(logits, 3)
    assert list(ids[0]) == [1, 4, 0]
    assert list(ids[1]) == [1, 3, 2]
    assert np.all(np.diff(w, axis=1) <= 0) and np.all(w.sum(axis=1) <= 1.0 + 1e-6)
    p = np.exp(logits[1] - 5.0) / np.exp(logits[1] - 5.0).sum()
    assert np.allclose(w[1], p[[1, 3, 2]], rtol=1e-6)


def test_permute_stable_brute_force():
    g = np.random.default_rng(25)
    ids = g.integers(0, 5, (7, 3)).astype(np.int32)
    offsets, perm = moe.permute(ids, 6)
    slots = sorted(range(21), key=lambda i: (ids.reshape(-1)[i], i))
    assert list(perm) == slots
    for e in range(6):
        assert offsets[e + 1] - offsets[e] == int((ids == e).sum())
    assert offsets[5] == offsets[6]         # expert 5 receives no rows


def _tiny_moe(seed, t, e, topk, hidden, inter, exact=True):
    g = synth.rng(seed)
    w1 = synth.expert_weights_fp32(g, e, hidden, 2 * inter)
    w2 = synth.expert_weights_fp32(g, e, inter, hidden)
    a = codecs.bf16(synth.activations_fp32(g, t, hidden))
    logits = synth.router_logits_fp32(g, t, e)
    w1h = [quant.dequant_int(*quant.quantize_int4_sym(w1[i], 32, "bf16"), None, 32, "bf16") for i in range(e)]
    w2h = [quant.dequant_int(*quant.quantize_int4_sym(w2[i], 32, "bf16"), None, 32, "bf16") for i in range(e)]
    ids, wts = moe.route(logits, topk)
    return a, ids, wts, w1h, w2h


def test_moe_layer_vs_per_token_brute_force():
    t, e, topk, hidden, inter = 5, 4, 2, 32, 32
    a, ids, wts, w1h, w2h = _tiny_moe(26, t, e, topk, hidden, inter)
    out = moe.moe_layer(a, ids, wts, lambda i: w1h[i], lambda i: w2h[i], e, inter)
    for tok in range(t):
        acc = np.zeros(hidden)
        for j in range(topk):
            ex = ids[tok, j]
            gu = codecs.bf16(np.array([math.fsum(a[tok, kk] * w1h[ex][kk, c] for kk in range(hidden))
                                       for c in range(2 * inter)]))
            gg, uu = gu[:inter], gu[inter:]
            h = codecs.bf16(gg / (1.0 + np.exp(-gg)) * uu)
            y2 = codecs.bf16(np.array([math.fsum(h[kk] * w2h[ex][kk, c] for kk in range(inter))
                                       for c in range(hidden)]))
            acc += float(wts[tok, j]) * y2
        assert np.array_equal(codecs.bf16(acc), out["y"][tok])


def test_moe_single_expert_reduces_to_two_dense_gemms():
    t, hidden, inter = 6, 64, 32
    a, _, _, w1h, w2h = _tiny_moe(27, t, 1, 1, hidden, inter)
    ids = np.zeros((t, 1), dtype=np.int32)
    wts = np.ones((t, 1), dtype=np.float32)
    out = moe.moe_layer(a, ids, wts, lambda i: w1h[i], lambda i: w2h[i], 1, inter)
    gu = codecs.bf16(a @ w1h[0])
    h = codecs.bf16(gu[:, :inter] / (1 + np.exp(-gu[:, :inter])) * gu[:, inter:])
    y = codecs.bf16(h @ w2h[0])
    assert np.array_equal(out["y"], y)
    assert list(out["perm"]) == list(range(t))
