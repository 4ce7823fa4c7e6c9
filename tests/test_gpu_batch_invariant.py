"""Batch-invariant mode on the GPU, through the C ABI: a row's output is
bitwise the same whatever the number and content of the other rows in the
call (dense: any m, any position of the row; grouped: any row counts of the
other experts), and every result stays within the oracle's tolerance.  The
heuristic picks the token tile by m, so the checks also cover a row computed
by tiles of different widths."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import DEV, TD, Case, assert_close, to_np
from oracle import codecs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


def _lin(c, **kw):
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    qw, sc, qz = c.dev_weights()
    return W4A16Linear(qw, sc, qz, c.n, c.k, c.g, TD[c.adt], bias=c.dev_bias(),
                       batch_invariant=True, **kw)


def _i16(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("sym,adt", [(True, "bf16"), (False, "fp16")])
def test_dense_rows_do_not_depend_on_m(Q, sym, adt, gated):
    if gated and adt != "bf16":
        pytest.skip("a gated output is bf16 only")
    c = Case(300, 384, 2048, 128, adt, sym, seed=91, bias=True)
    lin = _lin(c, gated=gated)
    x = c.dev_act()
    full = lin(x)
    assert lin.status() == Q.QGEMM_OK
    for m in (1, 3, 16, 17, 40, 64, 100, 129, 256):
        part = lin(x[:m].contiguous())
        assert torch.equal(_i16(part), _i16(full[:m])), f"m={m}"
    # the same rows at other positions of a differently composed batch
    perm = torch.from_numpy(np.random.default_rng(5).permutation(300)).to(DEV)
    shuffled = lin(x[perm].contiguous())
    assert torch.equal(_i16(shuffled), _i16(full[perm]))
    if not gated:
        assert_close(to_np(full), c.reference(), what="batch-invariant dense")


def test_grouped_rows_do_not_depend_on_other_experts(Q):
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    e, n, k, g = 4, 256, 1024, 128
    cases = [Case(1, n, k, g, "bf16", True, seed=300 + i) for i in range(e)]
    qw = torch.from_numpy(np.concatenate([cs.qweight for cs in cases])).to(DEV)
    sc = torch.from_numpy(np.concatenate([cs.s_bits for cs in cases]).view(np.int16)).to(DEV)
    lin = W4A16Linear(qw, sc, None, n, k, g, torch.bfloat16, num_experts=e,
                      batch_invariant=True)
    r = synth.rng(92)
    mine = codecs.bf16(synth.activations_fp32(r, 37, k))    # expert 2's rows, fixed
    outs = []
    for other in ([0, 0, 0], [5, 130, 1], [200, 3, 64], [1, 1, 900]):
        rows = [other[0], other[1], 37, other[2]]
        offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
        a = codecs.bf16(synth.activations_fp32(r, int(offsets[-1]), k))
        a[offsets[2]:offsets[3]] = mine
        out = lin.run_grouped(torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(DEV),
                              torch.from_numpy(offsets).to(DEV))
        assert lin.status() == Q.QGEMM_OK
        outs.append(out[offsets[2]:offsets[3]].clone())
        got = to_np(out)
        for i in range(e):
            r0, r1 = offsets[i], offsets[i + 1]
            if r1 > r0:
                assert_close(got[r0:r1], a[r0:r1] @ cases[i].w_hat, what=f"expert {i}")
    for o in outs[1:]:
        assert torch.equal(_i16(o), _i16(outs[0]))


def test_describe_plan_names_whole_tiles(Q):
    c = Case(8, 256, 256, 128, "bf16", True)
    lin = _lin(c)
    st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, 16)
    assert st == Q.QGEMM_OK and "split=whole_tiles" in rec
