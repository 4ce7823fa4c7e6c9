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
