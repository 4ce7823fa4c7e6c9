"""GPU parity of the small-M kernel (cp.async + mma.sync, K split over CTAs,
last-arrival finish), selected with tuning.kernel = 2, against the oracle:
|gpu - ref| <= 1e-2 + 1e-2 |ref| per element and relative Frobenius error
<= 5e-3, over M = 1..16, both 16-bit types, INT4 and UINT4, every group size,
bias, one and many K slices, repeated calls (the accumulators come back zero)
and the full-size M = 16 workloads; plus its rejections."""

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
    """Three calls in a row (the accumulators and counts are left at zero)
    agree with the oracle, and with the tcgen05 kernel within tolerance."""
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


def test_small_m_kernel_rejections(Q):
    c = Case(17, 256, 256, 128, "bf16", True)
    lin = _mma(Q, c)
    out = torch.empty(17, 256, dtype=torch.bfloat16, device=DEV)
    tun = Q.tuning_config(kernel=2)
    ws = lin.ws.get(1 << 20)
    # m > 16
    assert Q.qgemm_run(lin.layer, lin.dense, tun, 17, c.dev_act(), None, lin.packed, None, out,
                       ws, ws.numel()) == Q.QGEMM_ERR_UNSUPPORTED
    # deterministic compute
    det = Q.compute_config(Q.QGEMM_GEMM_DENSE, deterministic=1)
    st, _ = Q.qgemm_workspace_size(lin.layer, det, tun, 8)
    assert st == Q.QGEMM_ERR_UNSUPPORTED
    # unknown kernel id
    st, _ = Q.qgemm_workspace_size(lin.layer, lin.dense, Q.tuning_config(kernel=3), 8)
    assert st == Q.QGEMM_ERR_INVALID_ARG
