"""GPU parity of the tcgen05 kernel's cluster split (each output tile's K range
in S slices, one CTA per slice, the S CTAs of a tile in one thread-block
cluster summing their fp32 partials through distributed shared memory in
cluster-rank order), through the C ABI, against the oracle within the GEMM
tolerance of the other tests: every token tile size, cluster sizes 2 to 8
(powers of two and not), ragged M, more clusters than fit the device at once,
the 16-bit formats, W8A16, NVFP4 weights, W4A8, the gated epilogue and bias;
bitwise repeatability; the planner's choice; and the timeout path."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import DEV, TD, Case, assert_close, linear, to_np
from oracle import codecs, gemm, moe, quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


def _cl(Q, bt, s):
    return Q.tuning_config(block_tok=bt, split_k=s, kernel=3)


@pytest.mark.parametrize("bt", [16, 32, 64, 128])
@pytest.mark.parametrize("s", [2, 3, 4, 8])
def test_cluster_split_parity(Q, bt, s):
    m = {16: 13, 32: 45, 64: 70, 128: 200}[bt]
    c = Case(m, 384, 11 * 128, 128, "bf16", False, seed=bt + s)
    lin = linear(c, tuning=_cl(Q, bt, s))
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"cluster bt={bt} S={s}")
    st, plan = Q.qgemm_describe_plan(lin.layer, lin.dense, m)
    assert st == Q.QGEMM_OK


@pytest.mark.parametrize("adt,sym,g,bias", [("fp16", True, 128, False), ("bf16", False, 64, True),
                                            ("fp16", False, 32, True), ("bf16", True, 256, False)])
def test_cluster_split_formats_and_bias(Q, adt, sym, g, bias):
    c = Case(37, 256, 2048, g, adt, sym, seed=7, bias=bias)
    lin = linear(c, tuning=_cl(Q, 64, 4))
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"cluster {adt} sym={sym} g={g}")


def test_cluster_split_repeats_bitwise(Q):
    """The slices are summed in rank order, so two calls give the same bits."""
    c = Case(100, 512, 4096, 128, "bf16", False, seed=11)
    lin = linear(c, tuning=_cl(Q, 128, 4))
    x = c.dev_act()
    a = lin(x).clone()
    b = lin(x)
    assert lin.status() == Q.QGEMM_OK
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert_close(to_np(a), c.reference(), what="cluster repeat")


def test_cluster_split_more_clusters_than_fit(Q):
    """96 tiles x 4 slices = 384 CTAs of one SM each: the clusters run in
    several waves."""
    c = Case(300, 4096, 1024, 128, "bf16", True, seed=13)
    lin = linear(c, tuning=_cl(Q, 128, 4))
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what="cluster waves")


def test_cluster_split_gated(Q):
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    c = Case(45, 384, 2048, 128, "bf16", False, seed=17, bias=True)
    qw, sc, qz = c.dev_weights()
    lin = W4A16Linear(qw, sc, qz, c.n, c.k, c.g, TD[c.adt], bias=c.dev_bias(),
                      tuning=_cl(Q, 64, 4), gated=True)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    ref = moe.silu_mul(codecs.bf16(c.reference()), c.n // 2)
    assert_close(to_np(out), ref, what="cluster gated")


def test_cluster_split_w8a16(Q):
    from quantized_weight_gemm_run_b300.api import W8A16Linear
    r = synth.rng(19)
    m, n, k, g = 40, 256, 1536, 128
    w = synth.weights_fp32(r, k, n)
    a = codecs.bf16(synth.activations_fp32(r, m, k))
    q, s, z = quant.quantize_uint_asym(w, g, "bf16", 8)
    lin = W8A16Linear(torch.from_numpy(quant.pack_int_kn(q, 8, False)).to(DEV),
                      torch.from_numpy(codecs.dtype_bits("bf16", s).view(np.int16)).to(DEV),
                      torch.from_numpy(quant.pack_zeros_bits(z, 8)).to(DEV), n, k, g,
                      torch.bfloat16, tuning=_cl(Q, 64, 3))
    out = lin(torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(DEV))
    assert lin.status() == Q.QGEMM_OK
    ref = gemm.w4a16_reference(a, quant.dequant_int(q, s, z, g, "bf16"), None)
    assert_close(to_np(out), ref, what="cluster w8a16")


def test_cluster_split_w4a8(Q):
    from quantized_weight_gemm_run_b300.api import W4A8Linear
    r = synth.rng(23)
    m, n, k = 70, 384, 2048
    w = synth.weights_fp32(r, k, n)
    x = codecs.bf16(synth.activations_fp32(r, m, k))
    ckn, bkn = quant.quantize_mxfp4(w)
    cnk, bnk = quant.pack_mxfp4(ckn, bkn)
    lin = W4A8Linear(torch.from_numpy(cnk).to(DEV), torch.from_numpy(bnk).to(DEV), n, k,
                     tuning=_cl(Q, 128, 2))
    out = lin(torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(DEV))
    assert lin.status() == Q.QGEMM_OK
    a8, sc = gemm.act_quant_fp8(x)
    assert_close(to_np(out), gemm.w4a8_reference(a8, sc, ckn, bkn), frob=2e-2,
                 what="cluster w4a8")


def test_cluster_split_nvfp4(Q):
    from quantized_weight_gemm_run_b300.api import NVFP4Linear
    r = synth.rng(29)
    m, n, k = 33, 256, 1024
    w = synth.weights_fp32(r, k, n)
    x = codecs.bf16(synth.activations_fp32(r, m, k))
    codes, sb, ts = quant.quantize_nvfp4(w)
    cnk, snk = quant.pack_nvfp4(codes, sb)
    lin = NVFP4Linear(torch.from_numpy(cnk).to(DEV), torch.from_numpy(snk).to(DEV),
                      torch.tensor([ts], dtype=torch.float32, device=DEV), n, k, torch.bfloat16,
                      tuning=_cl(Q, 64, 4))
    out = lin(torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(DEV))
    assert lin.status() == Q.QGEMM_OK
    ref = gemm.w4a16_reference(x, quant.dequant_nvfp4(codes, sb, ts), None)
    assert_close(to_np(out), ref, what="cluster nvfp4")


@pytest.mark.parametrize("m,n,k", [(64, 4096, 4096), (256, 4096, 4096)])
def test_planner_takes_cluster_split_at_medium_m(Q, m, n, k):
    """The default plan of the medium-M sweep shapes whose tiles fit the device
    in clusters, and the parity of that default call."""
    c = Case(m, n, k, 128, "bf16", False, seed=m + n)
    lin = linear(c)
    st, plan = Q.qgemm_describe_plan(lin.layer, lin.dense, m)
    assert st == Q.QGEMM_OK
    assert "split=cluster_k" in plan, plan
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"default plan {m}x{n}x{k}")


def test_cluster_split_rejections(Q):
    c = Case(40, 256, 1024, 128, "bf16", True)
    for tun in (Q.tuning_config(kernel=3, split_k=9), Q.tuning_config(kernel=3, split_k=1),
                Q.tuning_config(kernel=3, block_tok=256),
                Q.tuning_config(kernel=3, max_ctas=10)):
        with pytest.raises(Q.QGemmError):
            linear(c, tuning=tun)(c.dev_act())
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    qw, sc, qz = c.dev_weights()
    lin = W4A16Linear(qw, sc, qz, c.n, c.k, c.g, TD[c.adt], tuning=Q.tuning_config(kernel=3),
                      batch_invariant=True)
    with pytest.raises(Q.QGemmError):
        lin(c.dev_act())


def test_cluster_split_timeout_reports_and_recovers(Q):
    """A wait limit of 0 makes the first unready wait give up: the status says
    timeout, every CTA still sends its slices and waits (bounded) for its own,
    the cluster leaves together, and the next call runs clean."""
    c = Case(70, 512, 2048, 128, "bf16", False, seed=31)
    lin = linear(c, tuning=_cl(Q, 64, 4))
    x = c.dev_act()
    ref = lin(x).clone()
    assert lin.status() == Q.QGEMM_OK
    Q.qgemm_set_wait_limit_ns(0)
    try:
        lin(x)
        torch.cuda.synchronize()
    finally:
        Q.qgemm_set_wait_limit_ns(1_000_000_000)
    assert lin.status() == Q.QGEMM_ERR_TIMEOUT
    lin.ws.get(256).zero_()
    again = lin(x)
    assert lin.status() == Q.QGEMM_OK
    torch.cuda.synchronize()
    assert torch.equal(again, ref)


def test_forced_cluster_split_without_a_count_takes_two_slices(Q):
    """kernel = 3 with split_k = 0 on a problem whose tiles alone fill the
    device: two slices per tile, in several waves."""
    c = Case(64, 11008, 1024, 128, "bf16", False, seed=41)
    lin = linear(c, tuning=Q.tuning_config(kernel=3))
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what="forced cluster, 86 tiles")
