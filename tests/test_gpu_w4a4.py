"""GPU parity of W4A4 (NVFP4 weights against NVFP4 activations on the FP4
tensor cores, tcgen05.mma kind::mxf4nvf4) through the C ABI, against the
oracle: the activation quantizer bit-exact (codes and block scales), the GEMM
within the GEMM tolerance of the other tests against the exact product of the
same quantized operands.  Structured operands (unit scales on one side, codes
and scales chosen per token and per 16-k block) separate the code, weight
scale and activation scale paths; every token tile size, ragged M, K spanning
more stages than the pipeline holds, bias, the timeout path and the
rejections.  The pages list W4A4 among the common configurations and name
NVFP4 (kinachrichten.com, "Warum quantisierte Kernel wichtig sind")."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import DEV, assert_close, to_np
from oracle import codecs, gemm, quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


def _bf16_dev(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(DEV)


def _f32_dev(v):
    return torch.tensor([v], dtype=torch.float32, device=DEV)


def _grid_acts(g, m, k, a_ts, unit_scales):
    """bf16 activations that quantize exactly to chosen codes and block scales:
    every block holds a +-6 code, so amax / (6 a_ts) is the block scale."""
    codes = g.integers(0, 16, size=(m, k)).astype(np.uint8)
    codes[codes == 8] = 0
    codes[:, ::16] = np.where(g.random((m, k // 16)) < 0.5, 0x7, 0xF)
    sb = (np.full((m, k // 16), 0x38, np.uint8) if unit_scales
          else g.integers(0x28, 0x48, size=(m, k // 16)).astype(np.uint8))
    x = gemm.nvfp4_act_operand(codes, sb) * a_ts
    assert np.array_equal(codecs.bf16(x), x)
    return x, codes, sb


def _weights(g, k, n, unit_scales, w_ts):
    codes = g.integers(0, 16, size=(k, n)).astype(np.uint8)
    sb = (np.full((k // 16, n), 0x38, np.uint8) if unit_scales
          else g.integers(0x20, 0x50, size=(k // 16, n)).astype(np.uint8))
    return codes, sb, w_ts


def _layer(codes_kn, sb_kn, w_ts, a_ts, n, k, bias=None, tuning=None):
    from quantized_weight_gemm_run_b300.api import W4A4Linear
    cnk, snk = quant.pack_nvfp4(codes_kn, sb_kn)
    return W4A4Linear(torch.from_numpy(cnk).to(DEV), torch.from_numpy(snk).to(DEV),
                      _f32_dev(w_ts), _f32_dev(a_ts), n, k,
                      bias=None if bias is None else _bf16_dev(bias), tuning=tuning)


def _check(Q, lin, x, a_ts, wc, wsb, w_ts, bias=None, what=""):
    out = lin(_bf16_dev(x))
    assert lin.status() == Q.QGEMM_OK
    ac, asb = gemm.act_quant_nvfp4(x, a_ts)
    ref = gemm.w4a4_reference(ac, asb, a_ts, wc, wsb, w_ts, bias)
    assert_close(to_np(out), ref, what=what)


@pytest.mark.parametrize("m,k,a_ts", [(1, 256, 1.0), (7, 512, 0.0123), (64, 1024, 2.0 ** -9),
                                      (130, 4096, 0.37)])
def test_act_quant_bit_exact(Q, m, k, a_ts):
    g = synth.rng(300 + m)
    x = codecs.bf16(synth.activations_fp32(g, m, k))
    x[0, :16] = 0.0                                   # an all-zero block
    x[-1, 16:32] *= 1e-30                             # a block whose scale rounds to zero
    if k >= 64:
        x[0, 48:64] *= 1e4                            # a saturating block
    codes = torch.empty(m, k // 2, dtype=torch.uint8, device=DEV)
    sb = torch.empty(m, k // 16, dtype=torch.uint8, device=DEV)
    Q.check(Q.qgemm_quantize_act_nvfp4(_bf16_dev(x), m, k, _f32_dev(a_ts), codes, sb))
    torch.cuda.synchronize()
    want_c, want_s = gemm.act_quant_nvfp4(x, a_ts)
    packed, _ = quant.pack_nvfp4(want_c.T, want_s.T)
    assert np.array_equal(sb.cpu().numpy(), want_s)
    got = codes.cpu().numpy()
    bad = np.argwhere(got != packed)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first at {bad[:4].tolist()}"


@pytest.mark.parametrize("w_unit,a_unit", [(True, True), (False, True), (True, False),
                                           (False, False)])
@pytest.mark.parametrize("m", [16, 40, 128])
def test_w4a4_structured_operands(Q, w_unit, a_unit, m):
    """Codes, weight block scales and activation block scales enter the MMA
    through separate paths: unit scales on one side isolate the other."""
    g = synth.rng(310 + m + 2 * w_unit + a_unit)
    n, k = 256, 512
    a_ts, w_ts = 0.5, 0.25
    x, _, _ = _grid_acts(g, m, k, a_ts, a_unit)
    wc, wsb, w_ts = _weights(g, k, n, w_unit, w_ts)
    lin = _layer(wc, wsb, w_ts, a_ts, n, k)
    _check(Q, lin, x, a_ts, wc, wsb, w_ts, what=f"w4a4 m={m} w_unit={w_unit} a_unit={a_unit}")


@pytest.mark.parametrize("bt", [16, 32, 64, 128])
@pytest.mark.parametrize("m", [1, 45, 200])
def test_w4a4_every_token_tile(Q, bt, m):
    g = synth.rng(320 + bt + m)
    n, k = 384, 768
    x = codecs.bf16(synth.activations_fp32(g, m, k))
    a_ts = float(np.float32(np.max(np.abs(x)) / (6 * 448)))
    wc, wsb, w_ts = quant.quantize_nvfp4(synth.weights_fp32(g, k, n))
    lin = _layer(wc, wsb, w_ts, a_ts, n, k, tuning=Q.tuning_config(block_tok=bt))
    _check(Q, lin, x, a_ts, wc, wsb, w_ts, what=f"w4a4 bt={bt} m={m}")


@pytest.mark.parametrize("m,n,k", [(256, 1024, 4096), (100, 512, 2048), (1, 4096, 4096)])
def test_w4a4_matches_oracle(Q, m, n, k):
    """Default plans; K of 8-16 stages runs the six-stage ring round more
    than once."""
    g = synth.rng(330 + m)
    x = codecs.bf16(synth.activations_fp32(g, m, k))
    a_ts = float(np.float32(np.max(np.abs(x)) / (6 * 448)))
    wc, wsb, w_ts = quant.quantize_nvfp4(synth.weights_fp32(g, k, n))
    bias = codecs.bf16(g.standard_normal(n))
    lin = _layer(wc, wsb, w_ts, a_ts, n, k, bias=bias)
    _check(Q, lin, x, a_ts, wc, wsb, w_ts, bias=bias, what=f"w4a4 {m}x{n}x{k}")


def test_w4a4_plan_and_rejections(Q):
    g = synth.rng(340)
    wc, wsb, w_ts = _weights(g, 512, 256, False, 1.0)
    lin = _layer(wc, wsb, w_ts, 1.0, 256, 512)
    # the M range's tile, or a smaller one while the tiles fit one wave (two
    # feature tiles here): 4096 rows in 64-token tiles are 128 tiles
    for m, bt in ((1, 16), (32, 32), (64, 32), (65, 32), (4096, 64), (8192, 128)):
        st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, m)
        assert st == Q.QGEMM_OK
        assert "kernel=w4a4_tcgen05_mxf4nvf4" in rec and f"block_tok={bt}" in rec, rec
    x = _bf16_dev(np.zeros((4, 512)))
    # k = 512 is two 256-k stages: at most two K slices
    for tun in (Q.tuning_config(split_k=3), Q.tuning_config(split_k=65),
                Q.tuning_config(kernel=2), Q.tuning_config(block_tok=256),
                Q.tuning_config(stages=3)):
        lin.tuning = tun
        with pytest.raises(Q.QGemmError):
            lin(x)
    lin.tuning = None
    # k not a multiple of 256, several experts, a gated output
    for kw in (dict(k=384), dict(num_experts=2), dict(gated_act=Q.QGEMM_ACT_SILU_GLU)):
        cfg = dict(n=256, k=512, group_size=16, weight_format=Q.QGEMM_W_NVFP4,
                   scale_format=Q.QGEMM_S_E4M3, zero_format=Q.QGEMM_Z_NONE,
                   act_dtype=Q.QGEMM_NVFP4, out_dtype=Q.QGEMM_BF16, has_bias=0, num_experts=1,
                   gated_act=Q.QGEMM_ACT_NONE)
        cfg.update(kw)
        st, _ = Q.qgemm_packed_size(Q.layer_config(**cfg))
        assert st == Q.QGEMM_ERR_UNSUPPORTED
    # the activation tensor scale is required
    ws = lin.ws.get(1 << 20)
    out = torch.empty(4, 256, dtype=torch.bfloat16, device=DEV)
    st = Q.qgemm_run(lin.layer, lin.dense, None, 4, x, None, lin.packed, None, out, ws,
                     ws.numel())
    assert st == Q.QGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("m,n,k,s", [(1, 512, 4096, 1), (1, 512, 4096, 4), (16, 384, 2560, 3),
                                     (45, 256, 3072, 5), (130, 256, 1024, 2), (7, 128, 512, 2)])
def test_w4a4_k_split(Q, m, n, k, s):
    """K slices of a tile summed by the last slice to count in: even and
    uneven slices, ragged M, bias, against the oracle."""
    g = synth.rng(360 + m + s)
    x = codecs.bf16(synth.activations_fp32(g, m, k))
    a_ts = float(np.float32(np.max(np.abs(x)) / (6 * 448)))
    wc, wsb, w_ts = quant.quantize_nvfp4(synth.weights_fp32(g, k, n))
    bias = codecs.bf16(g.standard_normal(n))
    lin = _layer(wc, wsb, w_ts, a_ts, n, k, bias=bias, tuning=Q.tuning_config(split_k=s))
    _check(Q, lin, x, a_ts, wc, wsb, w_ts, bias=bias, what=f"w4a4 split {s} {m}x{n}x{k}")


def test_w4a4_k_split_plan_repeats_and_reuses_workspace(Q):
    """The default plan splits K when the tiles leave SMs idle; the slices are
    summed in a fixed order (the bits repeat), and each call clears its own
    counters, so one workspace serves plans whose counters lie where another
    plan's partial tiles or quantized activations were."""
    g = synth.rng(370)
    n, k = 1024, 4096
    wc, wsb, w_ts = quant.quantize_nvfp4(synth.weights_fp32(g, k, n))
    xs = [codecs.bf16(synth.activations_fp32(g, m, k)) for m in (16, 300, 3)]
    a_ts = float(np.float32(max(np.max(np.abs(x)) for x in xs) / (6 * 448)))
    lin = _layer(wc, wsb, w_ts, a_ts, n, k)
    st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, 16)
    assert st == Q.QGEMM_OK and "split=k_slices_4_" in rec, rec   # 8 tiles, 16 stages
    st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, 8192)
    assert st == Q.QGEMM_OK and "split=whole_tiles" in rec, rec
    lin.ws.get(64 << 20)   # one workspace, large enough for every plan below
    first = {}
    for rnd in range(2):
        for x in xs:
            for tun in (None, Q.tuning_config(split_k=2), Q.tuning_config(split_k=16)):
                lin.tuning = tun
                out = lin(_bf16_dev(x))
                assert lin.status() == Q.QGEMM_OK
                key = (x.shape[0], None if tun is None else tun.split_k)
                got = to_np(out)
                if rnd == 0:
                    ac, asb = gemm.act_quant_nvfp4(x, a_ts)
                    ref = gemm.w4a4_reference(ac, asb, a_ts, wc, wsb, w_ts, None)
                    assert_close(got, ref, what=f"w4a4 reuse {key}")
                    first[key] = got
                else:
                    assert np.array_equal(got, first[key]), key


def test_w4a4_zero_rows_and_timeout(Q):
    g = synth.rng(350)
    n, k, m = 256, 1024, 33
    x = codecs.bf16(synth.activations_fp32(g, m, k))
    x[5] = 0.0
    a_ts = float(np.float32(np.max(np.abs(x)) / (6 * 448)))
    wc, wsb, w_ts = quant.quantize_nvfp4(synth.weights_fp32(g, k, n))
    lin = _layer(wc, wsb, w_ts, a_ts, n, k)
    xd = _bf16_dev(x)
    ref = lin(xd).clone()
    assert lin.status() == Q.QGEMM_OK
    assert not ref[5].any()
    Q.qgemm_set_wait_limit_ns(0)
    try:
        lin(xd)
        torch.cuda.synchronize()
    finally:
        Q.qgemm_set_wait_limit_ns(1_000_000_000)
    assert lin.status() == Q.QGEMM_ERR_TIMEOUT
    # no re-zeroing: each call clears the K split's counters (1 x 2 tiles here,
    # split across K), whatever an abandoned launch left in them
    again = lin(xd)
    assert lin.status() == Q.QGEMM_OK
    torch.cuda.synchronize()
    assert torch.equal(again, ref)
    empty = lin(xd[:0])
    assert empty.shape == (0, n)
