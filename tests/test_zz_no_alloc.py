"""The allocation-free dense GEMM entry point, qgemm_run_noalloc, through the
C ABI.  It serves callers that cannot allocate device memory when they run a
GEMM (code under an allocator lock it does not own, plugins inside a host
program that manages every device byte); it takes its split-K scratch from a
fixed array inside the library instead of a caller workspace.  Its output is
checked against the workspace entry point, qgemm_run, on two calls in a row
(the second call finds the scratch as the first one left it), within the
acceptance tolerance of the other GEMM tests.  This file is collected last on
purpose."""

import numpy as np
import pytest
import torch

from gpu_helpers import DEV, Case, assert_close, linear, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


@pytest.mark.parametrize("m,n,k,g,adt,sym", [
    (16, 4096, 4096, 128, "fp16", True),      # every tile split across CTAs
    (37, 384, 1024, 64, "bf16", False),       # ragged M, zero points
    (300, 640, 2048, 128, "bf16", True),      # several token tiles
])
def test_noalloc_matches_workspace_entry_point(Q, m, n, k, g, adt, sym):
    c = Case(m, n, k, g, adt, sym, seed=m + k)
    lin = linear(c)
    x = c.dev_act()
    ref_out = lin(x)                                       # qgemm_run, caller workspace
    assert lin.status() == Q.QGEMM_OK
    for _ in range(2):                                     # two calls in a row
        out = torch.full_like(ref_out, float("nan"))
        st = Q.qgemm_run_noalloc(lin.layer, lin.dense, None, m, x, None, lin.packed, None,
                                 out)
        assert st == Q.QGEMM_OK, Q.last_error()
        torch.cuda.synchronize()
        assert_close(to_np(out), to_np(ref_out), what="noalloc vs qgemm_run")
        assert_close(to_np(out), c.reference(), what="noalloc vs oracle")


def test_noalloc_second_plan_finds_its_scratch_clear(Q):
    """A split-K plan with a large scratch (the small-M kernel on 16x4096x4096:
    a count and a 16 x 128 accumulator per n-tile), then a different plan
    (the persistent kernel on a ragged 37-row problem), then the first again:
    each call must clear whatever the previous, different plan left."""
    cases = [Case(16, 4096, 4096, 128, "fp16", True, seed=5),
             Case(37, 384, 1024, 64, "bf16", False, seed=6)]
    lins = [linear(c) for c in cases]
    xs = [c.dev_act() for c in cases]
    refs = [lin(x) for lin, x in zip(lins, xs)]
    for lin in lins:
        assert lin.status() == Q.QGEMM_OK
    for i in (0, 1, 0, 1):
        c, lin, x = cases[i], lins[i], xs[i]
        out = torch.full_like(refs[i], float("nan"))
        st = Q.qgemm_run_noalloc(lin.layer, lin.dense, None, c.m, x, None, lin.packed, None, out)
        assert st == Q.QGEMM_OK, Q.last_error()
        assert Q.qgemm_noalloc_check_status() == Q.QGEMM_OK
        assert_close(to_np(out), to_np(refs[i]), what=f"noalloc plan {i} vs qgemm_run")


def test_noalloc_reports_a_timeout_and_recovers(Q):
    """A wait limit of 0 makes the persistent kernel's first unready wait give
    up (it records the status, drains its copies and exits: no fault, no
    hang).  A call rejected by an argument check in between must queue
    nothing, so the status word it would otherwise have cleared still says
    timeout; the status call reports it, and the next call runs clean."""
    c = Case(40, 256, 1024, 128, "bf16", True, seed=3)
    lin = linear(c)
    x = c.dev_act()
    ref = lin(x)
    assert lin.status() == Q.QGEMM_OK
    out = torch.empty_like(ref)
    Q.qgemm_set_wait_limit_ns(0)
    try:
        st = Q.qgemm_run_noalloc(lin.layer, lin.dense, None, c.m, x, None, lin.packed, None, out)
        assert st == Q.QGEMM_OK, Q.last_error()
        torch.cuda.synchronize()
    finally:
        Q.qgemm_set_wait_limit_ns(1_000_000_000)
    st = Q.qgemm_run_noalloc(lin.layer, lin.dense, None, c.m, x.data_ptr() + 2, None,
                             lin.packed, None, out)            # misaligned: rejected
    assert st == Q.QGEMM_ERR_INVALID_ARG
    assert Q.qgemm_noalloc_check_status() == Q.QGEMM_ERR_TIMEOUT
    st = Q.qgemm_run_noalloc(lin.layer, lin.dense, None, c.m, x, None, lin.packed, None, out)
    assert st == Q.QGEMM_OK, Q.last_error()
    assert Q.qgemm_noalloc_check_status() == Q.QGEMM_OK
    assert_close(to_np(out), to_np(ref), what="noalloc after a timeout")


def test_noalloc_rejects_problems_beyond_its_scratch(Q):
    # 2^20 rows x 16384 columns needs more split-K counters than 32 MiB holds
    layer = Q.layer_config(16384, 4096, 128, Q.QGEMM_W_INT4_SYM, Q.QGEMM_S_BF16, Q.QGEMM_Z_NONE,
                           Q.QGEMM_BF16, Q.QGEMM_BF16)
    dense = Q.compute_config(Q.QGEMM_GEMM_DENSE)
    dummy = torch.zeros(16, dtype=torch.uint8, device=DEV)
    st = Q.qgemm_run_noalloc(layer, dense, None, 1 << 20, dummy, None, dummy, None, dummy)
    assert st == Q.QGEMM_ERR_UNSUPPORTED
    assert "scratch" in Q.last_error()


def test_noalloc_refuses_grouped(Q):
    layer = Q.layer_config(256, 256, 128, Q.QGEMM_W_INT4_SYM, Q.QGEMM_S_BF16, Q.QGEMM_Z_NONE,
                           Q.QGEMM_BF16, Q.QGEMM_BF16, num_experts=4)
    st = Q.qgemm_run_noalloc(layer, Q.compute_config(Q.QGEMM_GEMM_GROUPED), None, 8, 16, None,
                             16, None, 16)
    assert st == Q.QGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("m", [5, 70])
def test_noalloc_w4a8_on_bf16_activations(Q, m):
    """W4A8 layers on bf16 activations through the allocation-free entry point:
    at m <= 8 the quantization runs inside the small-M kernel, above it the
    quantized rows and scales live in the library's scratch (after the part
    that is cleared) before the tcgen05 kernel reads them."""
    import synth
    from oracle import codecs, quant
    from quantized_weight_gemm_run_b300.api import W4A8Linear
    g = synth.rng(40 + m)
    n, k = 384, 1024
    ckn, bkn = quant.quantize_mxfp4(synth.weights_fp32(g, k, n))
    cnk, bnk = quant.pack_mxfp4(ckn, bkn)
    lin = W4A8Linear(torch.from_numpy(cnk).to(DEV), torch.from_numpy(bnk).to(DEV), n, k)
    x = torch.from_numpy(codecs.bf16(synth.activations_fp32(g, m, k)).astype(np.float32)).to(
        torch.bfloat16).to(DEV)
    ref = lin(x)
    assert lin.status() == Q.QGEMM_OK
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        st = Q.qgemm_run_noalloc(lin.layer_bf16, lin.dense, None, m, x, None, lin.packed, None,
                                 out)
        assert st == Q.QGEMM_OK, Q.last_error()
        assert Q.qgemm_noalloc_check_status() == Q.QGEMM_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref)


@pytest.mark.parametrize("m,n,k", [(16, 512, 4096), (300, 384, 1024)])
def test_noalloc_w4a4(Q, m, n, k):
    """W4A4 layers through the allocation-free entry point: the NVFP4 codes and
    block scales of the activations, and (at m = 16, a K split) the slices'
    partial tiles live in the library's scratch; the K split's counters are
    cleared by the call's own quantization kernel, so the bits equal the
    workspace entry point's on two calls in a row."""
    import synth
    from oracle import codecs, quant
    from quantized_weight_gemm_run_b300.api import W4A4Linear
    g = synth.rng(60 + m)
    wc, wsb, w_ts = quant.quantize_nvfp4(synth.weights_fp32(g, k, n))
    cnk, snk = quant.pack_nvfp4(wc, wsb)
    x32 = codecs.bf16(synth.activations_fp32(g, m, k))
    a_ts = torch.tensor([float(np.float32(np.max(np.abs(x32)) / (6 * 448)))],
                        dtype=torch.float32, device=DEV)
    lin = W4A4Linear(torch.from_numpy(cnk).to(DEV), torch.from_numpy(snk).to(DEV),
                     torch.tensor([w_ts], dtype=torch.float32, device=DEV), a_ts, n, k)
    x = torch.from_numpy(x32.astype(np.float32)).to(torch.bfloat16).to(DEV)
    ref = lin(x)
    assert lin.status() == Q.QGEMM_OK
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        st = Q.qgemm_run_noalloc(lin.layer, lin.dense, None, m, x, lin.act_scale, lin.packed,
                                 None, out)
        assert st == Q.QGEMM_OK, Q.last_error()
        assert Q.qgemm_noalloc_check_status() == Q.QGEMM_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
