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


@pytest.mark.parametrize("m", [1, 5, 8, 9, 16])
@pytest.mark.parametrize("bias", [False, True])
def test_w4a8_small_m_kernel_matches_oracle_and_tcgen05(Q, m, bias):
    """M <= 16 runs on the small-M kernel (e4m3 register MMAs, the e8m0 scale
    applied per 32-k partial); the tcgen05 kernel forced on the same problem
    gives the same result within tolerance."""
    from quantized_weight_gemm_run_b300.api import W4A8Linear
    c = MxCase(m, 640, 2048, seed=61 + m)
    bvec = None
    if bias:
        bvec = codecs.bf16(synth.rng(62).standard_normal(c.n) * 0.5)
    bdev = None if bvec is None else torch.from_numpy(bvec.astype(np.float32)).to(
        torch.bfloat16).to(DEV)
    lin2 = W4A8Linear(torch.from_numpy(c.codes_nk).to(DEV), torch.from_numpy(c.b_nk).to(DEV),
                      c.n, c.k, bias=bdev, tuning=Q.tuning_config(kernel=2))
    lin1 = W4A8Linear(torch.from_numpy(c.codes_nk).to(DEV), torch.from_numpy(c.b_nk).to(DEV),
                      c.n, c.k, bias=bdev, tuning=Q.tuning_config(kernel=1))
    x = c.x_dev()
    ref = c.reference() + (0 if bvec is None else bvec[None, :])
    out2 = lin2(x)
    assert lin2.status() == Q.QGEMM_OK
    assert_close(to_np(out2), ref, frob=2e-2, what=f"w4a8 small-M kernel m={m}")
    out1 = lin1(x)
    assert lin1.status() == Q.QGEMM_OK
    assert_close(to_np(out2), to_np(out1), frob=2e-2, what=f"w4a8 kernels agree m={m}")


@pytest.mark.parametrize("split_k", [1, 2, 4, 8, 16])
def test_w4a8_small_m_cluster_sizes(Q, split_k):
    from quantized_weight_gemm_run_b300.api import W4A8Linear
    c = MxCase(11, 384, 21 * 128, seed=70 + split_k)
    lin = W4A8Linear(torch.from_numpy(c.codes_nk).to(DEV), torch.from_numpy(c.b_nk).to(DEV),
                     c.n, c.k, tuning=Q.tuning_config(kernel=2, split_k=split_k))
    out = lin(c.x_dev())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), frob=2e-2, what=f"w4a8 S={split_k}")


def test_w4a8_small_m_every_code_and_wide_scales(Q):
    """Every e2m1 code in every nibble position and block scales from 2^-27 to
    2^27 through the small-M kernel's own conversion and scale path."""
    from quantized_weight_gemm_run_b300.api import W4A8Linear
    n, k, m = 256, 512, 3
    codes = np.tile(np.arange(16, dtype=np.uint8), (k * n) // 16).reshape(k, n)
    codes = np.roll(codes, 5, axis=1)
    r = synth.rng(71)
    b = r.integers(100, 155, size=(k // 32, n)).astype(np.uint8)
    cn, bn = quant.pack_mxfp4(codes, b)
    x = codecs.bf16(synth.activations_fp32(r, m, k))
    lin = W4A8Linear(torch.from_numpy(cn).to(DEV), torch.from_numpy(bn).to(DEV), n, k,
                     tuning=Q.tuning_config(kernel=2))
    out = lin(torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(DEV))
    assert lin.status() == Q.QGEMM_OK
    a8, s = gemm.act_quant_fp8(x)
    assert_close(to_np(out), gemm.w4a8_reference(a8, s, codes, b), frob=2e-2,
                 what="w4a8 every code, wide scales")


# ---- bf16 activations quantized by the library (one call)

def _lin(Q, c, **tuning):
    from quantized_weight_gemm_run_b300.api import W4A8Linear
    t = Q.tuning_config(**tuning) if tuning else None
    return W4A8Linear(torch.from_numpy(c.codes_nk).to(DEV), torch.from_numpy(c.b_nk).to(DEV),
                      c.n, c.k, tuning=t)


@pytest.mark.parametrize("m", [1, 3, 8, 9, 16, 17, 70])
def test_w4a8_one_call_bitwise_equals_two_calls(Q, m):
    """The one-call form on bf16 activations (quantized inside the small-M
    kernel at m <= 8, by the quantizer kernel into the workspace above) gives
    the same bits as qgemm_quantize_act_fp8 followed by qgemm_run: the
    quantization is the same arithmetic, the maximum over the K slices is
    exact, and the GEMM then reads the same codes and scales."""
    c = MxCase(m, 640, 2048, seed=80 + m)
    lin = _lin(Q, c)
    x = c.x_dev()
    one = lin(x)
    assert lin.status() == Q.QGEMM_OK
    two = lin.two_call(x)
    assert lin.status() == Q.QGEMM_OK
    torch.cuda.synchronize()
    assert torch.equal(one, two), f"m={m}: one-call and two-call results differ"
    assert_close(to_np(one), c.reference(), frob=2e-2, what=f"w4a8 one call m={m}")
    st, plan = Q.qgemm_describe_plan(lin.layer_bf16, lin.dense, m)
    assert st == Q.QGEMM_OK
    assert ("act_quant=fused" if m <= 8 else "act_quant=separate_kernel") in plan, plan


@pytest.mark.parametrize("split_k", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("m", [2, 13])
def test_w4a8_fused_quant_cluster_sizes(Q, split_k, m):
    """Every cluster size of the small-M kernel: each CTA sees a different K
    slice, so a row's scale needs the maxima of all S slices (a slice that
    ends in the tail k-tiles of a 21-tile K included)."""
    c = MxCase(m, 384, 21 * 128, seed=90 + split_k + m)
    # one row's largest |x| placed in the last slice only, another's in the first
    c.x[0, :] *= 0.01
    c.x[0, -5] = 37.0
    if m > 1:
        c.x[1, :] *= 0.01
        c.x[1, 3] = -29.0
    lin = _lin(Q, c, kernel=2, split_k=split_k)
    x = c.x_dev()
    one = lin(x)
    assert lin.status() == Q.QGEMM_OK
    two = lin.two_call(x)
    torch.cuda.synchronize()
    assert torch.equal(one, two), f"S={split_k} m={m}"
    assert_close(to_np(one), c.reference(), frob=2e-2, what=f"fused quant S={split_k} m={m}")


def test_w4a8_fused_quant_zero_and_saturating_rows(Q):
    """An all-zero row (scale 1, every code 0) and rows whose values span the
    e4m3 range up to the row maximum (code 448) through the fused path."""
    m = 6
    c = MxCase(m, 256, 1024, seed=95)
    c.x[2, :] = 0.0
    c.x[4, :] = codecs.bf16(np.linspace(-3e4, 3e4, c.k))
    c.x[5, :] = codecs.bf16(np.full(c.k, 1e-30))
    lin = _lin(Q, c, kernel=2)
    x = c.x_dev()
    one = lin(x)
    assert lin.status() == Q.QGEMM_OK
    two = lin.two_call(x)
    torch.cuda.synchronize()
    assert torch.equal(one, two)
    assert np.all(to_np(one)[2] == 0.0)
    assert_close(to_np(one), c.reference(), frob=2e-2, what="fused quant edge rows")


def test_w4a8_fused_quant_timeout_reports_and_recovers(Q):
    """A wait limit of 0 makes the small-M kernel's waits (the activation box,
    the slices' maxima, the partial sums) give up: the status says timeout,
    every CTA drains within its bounded waits, and the next call runs clean."""
    c = MxCase(5, 512, 2048, seed=97)
    lin = _lin(Q, c, kernel=2)
    x = c.x_dev()
    ref = lin(x)
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


def test_w4a8_bf16_rejects_caller_scales(Q):
    c = MxCase(4, 128, 128, seed=98)
    lin = _lin(Q, c)
    x = c.x_dev()
    sc = torch.ones(4, dtype=torch.float32, device=DEV)
    out = torch.empty(4, 128, dtype=torch.bfloat16, device=DEV)
    st, need = Q.qgemm_workspace_size(lin.layer_bf16, lin.dense, None, 4)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    assert Q.qgemm_run(lin.layer_bf16, lin.dense, None, 4, x, sc, lin.packed, None, out,
                       ws, need) == Q.QGEMM_ERR_INVALID_ARG


def test_w4a8_bf16_grouped_matches_per_expert(Q):
    """Grouped W4A8 on bf16 activations: the quantizer kernel runs over all
    rows, then the grouped tcgen05 kernel; each expert's rows match the dense
    two-call form of that expert."""
    from quantized_weight_gemm_run_b300.api import W4A8Linear
    e, n, k = 3, 256, 512
    cs = [MxCase(1, n, k, seed=100 + i) for i in range(e)]
    codes = torch.from_numpy(np.concatenate([c.codes_nk for c in cs])).to(DEV)
    bs = torch.from_numpy(np.concatenate([c.b_nk for c in cs])).to(DEV)
    lin = W4A8Linear(codes, bs, n, k, num_experts=e)
    rows = [5, 0, 40]
    offs = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    x = codecs.bf16(synth.activations_fp32(synth.rng(104), int(offs[-1]), k))
    xd = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(DEV)
    out = torch.empty(int(offs[-1]), n, dtype=torch.bfloat16, device=DEV)
    st, need = Q.qgemm_workspace_size(lin.layer_bf16, lin.grouped, None, int(offs[-1]))
    assert st == Q.QGEMM_OK
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    od = torch.from_numpy(offs).to(DEV)
    assert Q.qgemm_grouped_run(lin.layer_bf16, lin.grouped, None, od, int(offs[-1]), xd, None,
                               lin.packed, None, out, ws, need) == Q.QGEMM_OK, Q.last_error()
    assert Q.qgemm_check_status(ws) == Q.QGEMM_OK
    got = to_np(out)
    for i, c in enumerate(cs):
        lo, hi = offs[i], offs[i + 1]
        if hi == lo:
            continue
        a8, s = gemm.act_quant_fp8(x[lo:hi])
        want = gemm.w4a8_reference(a8, s, c.codes_kn, c.b_kn)
        assert_close(got[lo:hi], want, frob=2e-2, what=f"grouped w4a8 bf16 expert {i}")


def test_w4a8_bf16_one_workspace_across_plans(Q):
    """A layer on bf16 activations keeps its quantized rows in the workspace,
    at an offset that depends on the plan.  Calls that switch plans on one
    workspace (the cluster split and the small-M kernel put the rows where a
    stream-K plan keeps its split-K counters and accumulator) must each give
    the right result: the stream-K plan, which only a tuning selects for these
    layers, clears its state first."""
    c = MxCase(64, 1024, 2048, seed=120)
    lin = _lin(Q, c)
    x = c.x_dev()
    ref = c.reference()
    plans = {"cluster": (64, Q.tuning_config(kernel=3, split_k=2)),
             "stream_k": (64, Q.tuning_config(block_tok=32, max_ctas=37)),
             "small_m": (16, Q.tuning_config(kernel=2)),
             "default": (64, None)}
    need = max(Q.qgemm_workspace_size(lin.layer_bf16, lin.dense, t, m)[1] for m, t in plans.values())
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for name in ("stream_k", "cluster", "stream_k", "small_m", "stream_k", "default", "stream_k"):
        m, tun = plans[name]
        out = torch.full((m, c.n), float("nan"), dtype=torch.bfloat16, device=DEV)
        st = Q.qgemm_run(lin.layer_bf16, lin.dense, tun, m, x[:m].contiguous(), None, lin.packed,
                         None, out, ws, need)
        assert st == Q.QGEMM_OK, (name, Q.last_error())
        assert Q.qgemm_check_status(ws) == Q.QGEMM_OK, (name, Q.last_error())
        assert_close(to_np(out), ref[:m], frob=2e-2, what=f"w4a8 plan {name}")


@pytest.mark.parametrize("m", [100, 256, 512])
def test_w4a8_planner_takes_whole_tiles(Q, m):
    c = MxCase(m, 7168, 2048, seed=130 + m)
    lin = _lin(Q, c)
    st, plan = Q.qgemm_describe_plan(lin.layer_bf16, lin.dense, m)
    assert st == Q.QGEMM_OK
    assert "split=whole_tiles" in plan or "split=cluster" in plan, plan
    if m == 100:
        assert "block_tok=64" in plan, plan
    out = lin(c.x_dev())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), frob=2e-2, what=f"w4a8 m={m}")
