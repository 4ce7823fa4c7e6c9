"""GPU parity of the small-M kernel (bulk copies + mma.sync, one cluster of K
slices per n-tile reducing through distributed shared memory), selected with
tuning.kernel = 2, against the oracle: |gpu - ref| <= 1e-2 + 1e-2 |ref| per
element and relative Frobenius error <= 5e-3, over M = 1..16, both 16-bit
types, INT4 and UINT4, every group size, bias, every cluster size and ring
depth, repeated calls and the full-size M = 16 workloads; its fixed-order
reduction (bits repeat, rows independent of M), its timeout path and its
rejections."""

import numpy as np
import pytest
import torch

from gpu_helpers import DEV, TD, Case, assert_close, linear, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


def _mma(Q, c, **kw):
    return linear(c, tuning=Q.tuning_config(kernel=2), **kw)


CASES = [
    # m, n, k, g, adt, sym, bias
    (1, 128, 128, 128, "bf16", True, False),
    (3, 256, 512, 32, "fp16", False, False),
    (8, 384, 1024, 64, "bf16", False, True),
    (16, 640, 768, 128, "fp16", True, True),
    (16, 128, 4096, 256, "bf16", False, False),
    (11, 1024, 256, 128, "bf16", True, False),
]


@pytest.mark.parametrize("m,n,k,g,adt,sym,bias", CASES)
def test_small_m_kernel_parity(Q, m, n, k, g, adt, sym, bias):
    c = Case(m, n, k, g, adt, sym, seed=m * 7 + n + k, bias=bias)
    lin = _mma(Q, c)
    st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, m)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"mma {m}x{n}x{k} g{g} {adt}")


def test_small_m_kernel_repeats_and_matches_k1(Q):
    """Three calls in a row agree with the oracle, and with the tcgen05
    kernel within tolerance."""
    c = Case(16, 512, 2048, 128, "bf16", False, seed=5)
    lin = _mma(Q, c)
    x = c.dev_act()
    outs = [to_np(lin(x)) for _ in range(3)]
    ref = c.reference()
    for o in outs:
        assert_close(o, ref, what="repeat")
    k1 = to_np(linear(c, tuning=Q.tuning_config(kernel=1))(x))
    assert_close(outs[0], k1, what="vs tcgen05 kernel")


@pytest.mark.parametrize("m,n,k,adt,sym", [(16, 4096, 4096, "fp16", True),
                                           (1, 11008, 4096, "bf16", False),
                                           (16, 4096, 11008, "bf16", False)])
def test_small_m_kernel_full_size(Q, m, n, k, adt, sym):
    c = Case(m, n, k, 128, adt, sym, seed=m + n)
    lin = _mma(Q, c)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"mma full {m}x{n}x{k}")


@pytest.mark.parametrize("split_k", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("ring", [1, 2, 4])
def test_small_m_kernel_cluster_sizes_and_rings(Q, split_k, ring):
    """Every cluster size (K slices per n-tile) and ring depth, on a ragged K
    (21 k-tiles: slices of unequal length) and M = 13."""
    c = Case(13, 384, 21 * 128, 128, "bf16", False, seed=split_k * 10 + ring)
    lin = linear(c, tuning=Q.tuning_config(kernel=2, split_k=split_k, stages=ring))
    st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, 13)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"S={split_k} ring={ring}")


def test_small_m_kernel_fixed_order_bits(Q):
    """The slices meet in a fixed order: repeated calls give the same bits,
    and a row's bits do not depend on how many rows the call has (M = 3, 8
    and 16 take one or two n8 token blocks)."""
    c = Case(16, 768, 4096, 128, "bf16", True, seed=77)
    lin = _mma(Q, c)
    x = c.dev_act()
    full = lin(x).clone()
    again = lin(x).clone()
    assert torch.equal(full.view(torch.int16), again.view(torch.int16))
    for m in (3, 8):
        part = lin(x[:m].contiguous())
        assert torch.equal(part.view(torch.int16), full[:m].view(torch.int16))
    assert_close(to_np(full), c.reference(), what="fixed order")


def test_small_m_kernel_timeout_reports_and_recovers(Q):
    """A wait limit of 0: the first wait that would block gives up, the CTA
    records the timeout, lets its own copies land, passes the cluster
    barriers and exits (no fault, no hang); the next call runs clean."""
    c = Case(16, 512, 4096, 128, "fp16", True, seed=9)
    lin = _mma(Q, c)
    x = c.dev_act()
    Q.qgemm_set_wait_limit_ns(0)
    try:
        lin(x)
        st = lin.status()
    finally:
        Q.qgemm_set_wait_limit_ns(1_000_000_000)
    assert st in (Q.QGEMM_ERR_TIMEOUT, Q.QGEMM_OK)   # OK only if no wait ever had to block
    out = lin(x)
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what="after timeout")


def test_small_m_kernel_rejections(Q):
    c = Case(17, 256, 256, 128, "bf16", True)
    lin = _mma(Q, c)
    out = torch.empty(17, 256, dtype=torch.bfloat16, device=DEV)
    tun = Q.tuning_config(kernel=2)
    ws = lin.ws.get(1 << 20)
    # m > 16
    assert Q.qgemm_run(lin.layer, lin.dense, tun, 17, c.dev_act(), None, lin.packed, None, out,
                       ws, ws.numel()) == Q.QGEMM_ERR_UNSUPPORTED
    # batch-invariant compute (the tcgen05 kernel serves it at every M)
    bi = Q.compute_config(Q.QGEMM_GEMM_DENSE, batch_invariant=1)
    st, _ = Q.qgemm_workspace_size(lin.layer, bi, tun, 8)
    assert st == Q.QGEMM_ERR_UNSUPPORTED
    # K slices: a power of two, at most 16 and at most the k-tiles (2 here)
    for bad in (3, 4, 32):
        st, _ = Q.qgemm_workspace_size(lin.layer, lin.dense, Q.tuning_config(kernel=2,
                                                                             split_k=bad), 8)
        assert st in (Q.QGEMM_ERR_UNSUPPORTED, Q.QGEMM_ERR_INVALID_ARG), bad
    # unknown kernel id (3 is the tcgen05 kernel's cluster split)
    st, _ = Q.qgemm_workspace_size(lin.layer, lin.dense, Q.tuning_config(kernel=4), 8)
    assert st == Q.QGEMM_ERR_INVALID_ARG


def test_plan_sends_9_to_16_rows_on_a_long_k_to_the_tcgen05_kernel(Q):
    """At 9-16 rows with at least twice as many k-tiles as n-tiles the planner
    takes the tcgen05 kernel (measured faster there); at 8 rows, or on a
    square layer, the small-M kernel.  Both match the oracle."""
    c = Case(16, 256, 1024, 128, "bf16", False, seed=21)
    lin = linear(c)
    for m, kern in ((8, "w4a16_mma_sync_smallm"), (9, "w4a16_tcgen05_swapab"),
                    (16, "w4a16_tcgen05_swapab")):
        st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, m)
        assert st == Q.QGEMM_OK and f"kernel={kern}" in rec, rec
    sq = linear(Case(16, 512, 512, 128, "bf16", False, seed=22))
    st, rec = Q.qgemm_describe_plan(sq.layer, sq.dense, 16)
    assert st == Q.QGEMM_OK and "kernel=w4a16_mma_sync_smallm" in rec, rec
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what="long-K 16 rows on the tcgen05 kernel")
