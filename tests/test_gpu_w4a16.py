"""GPU parity of the W4A16 path against the oracle, through the C ABI: the
repack and the dequantization bit for bit, the GEMM within the acceptance
tolerance (|gpu - ref| <= 1e-2 + 1e-2 |ref| per element, relative Frobenius
error <= 5e-3), at small sizes spanning several tiles and a ragged M tail, at
the full workload sizes, and on the edge and error cases."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import DEV, TD, Case, assert_close, linear, to_np
from oracle import codecs, layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


@pytest.mark.parametrize("adt,sym,g", [("bf16", True, 128), ("fp16", True, 32),
                                       ("bf16", False, 64), ("bf16", False, 256),
                                       ("fp16", False, 128)])
def test_repack_and_dequant_bit_exact(Q, adt, sym, g):
    c = Case(8, 384, 512, g, adt, sym, seed=31)
    lin = linear(c)
    torch.cuda.synchronize()
    want = layout.packed_w4(c.q, c.s_bits, c.z, g, signed=sym)
    assert np.array_equal(lin.packed.cpu().numpy(), want)
    deq = lin.dequantized().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, codecs.dtype_bits(adt, c.w_hat))


SMALL = [
    # m, n, k, g, adt, sym
    (1, 128, 128, 128, "bf16", True),
    (16, 128, 256, 128, "bf16", True),
    (37, 384, 512, 128, "bf16", False),
    (37, 384, 512, 128, "fp16", True),
    (5, 256, 1024, 64, "bf16", False),
    (200, 256, 512, 32, "fp16", True),
    (129, 256, 384, 128, "bf16", False),
    (64, 512, 256, 256, "bf16", True),
    (300, 640, 1024, 128, "fp16", False),
]


@pytest.mark.parametrize("m,n,k,g,adt,sym", SMALL)
def test_gemm_small_parity(Q, m, n, k, g, adt, sym):
    c = Case(m, n, k, g, adt, sym, seed=m + n + k)
    lin = linear(c)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"{m}x{n}x{k}")


def test_gemm_bias(Q):
    c = Case(21, 256, 384, 128, "bf16", False, seed=5, bias=True)
    lin = linear(c)
    out = lin(c.dev_act())
    assert_close(to_np(out), c.reference(), what="bias")


@pytest.mark.parametrize("det", [False, True])
@pytest.mark.parametrize("bt", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("split_k,max_ctas", [(0, 0), (1, 0), (0, 7)])
def test_tuning_overrides_same_result(Q, bt, split_k, max_ctas, det):
    c = Case(70, 384, 768, 128, "bf16", False, seed=9)
    lin = linear(c, tuning=Q.tuning_config(block_tok=bt, split_k=split_k, max_ctas=max_ctas),
                 deterministic=det)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"bt={bt} split_k={split_k} ctas={max_ctas}")


@pytest.mark.parametrize("m,adt,sym,split_k,max_ctas", [
    (600, "bf16", True, 0, 0),      # ragged last 256-token tile, stream-K
    (600, "fp16", False, 1, 0),     # whole tiles
    (1024, "bf16", False, 0, 5),    # few CTAs: long stream-K ranges
])
def test_256_token_tiles(Q, m, adt, sym, split_k, max_ctas):
    """The 256-token tile (one 256-column accumulator, N = 256 MMAs) over
    several token tiles, a ragged last tile, split and whole tiles."""
    c = Case(m, 640, 1536, 128, adt, sym, seed=m + 3)
    lin = linear(c, tuning=Q.tuning_config(block_tok=256, split_k=split_k, max_ctas=max_ctas))
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"bt=256 m={m} {adt}")


def test_256_token_tiles_reject_other_formats(Q):
    layer = Q.layer_config(256, 256, 32, Q.QGEMM_W_MXFP4, Q.QGEMM_S_E8M0, Q.QGEMM_Z_NONE,
                           Q.QGEMM_FP8E4M3, Q.QGEMM_BF16)
    st, _ = Q.qgemm_workspace_size(layer, Q.compute_config(Q.QGEMM_GEMM_DENSE),
                                   Q.tuning_config(block_tok=256), 512)
    assert st == Q.QGEMM_ERR_UNSUPPORTED


def test_deterministic_mode_bits_repeat(Q):
    c = Case(48, 512, 2048, 128, "bf16", True, seed=12)
    lin = linear(c, tuning=Q.tuning_config(max_ctas=37), deterministic=True)   # many split tiles
    x = c.dev_act()
    o1 = lin(x).clone()
    o2 = lin(x).clone()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert_close(to_np(o1), c.reference(), what="deterministic mode")


def test_atomic_mode_repeats_within_tolerance(Q):
    c = Case(48, 512, 2048, 128, "bf16", True, seed=12)
    lin = linear(c, tuning=Q.tuning_config(max_ctas=37))
    x = c.dev_act()
    outs = [to_np(lin(x)) for _ in range(3)]   # accumulators must come back zeroed each time
    for o in outs:
        assert_close(o, c.reference(), what="atomic split-K")


def test_m_zero_launches_nothing(Q):
    c = Case(4, 128, 128, 128, "bf16", True)
    lin = linear(c)
    x = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    st, ws_bytes = Q.qgemm_workspace_size(lin.layer, lin.dense, None, 1)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
    assert Q.qgemm_run(lin.layer, lin.dense, None, 0, x, None, lin.packed, None, out,
                       ws, ws_bytes) == Q.QGEMM_OK


def test_full_size_w4a16_sym_m16(Q):
    s = synth.W4A16_SYM_SHAPE
    c = Case(s["m"], s["n"], s["k"], s["group"], "fp16", True, seed=synth.SEED_W4A16_SYM)
    lin = linear(c)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what="M=16 4096x4096 fp16")


@pytest.mark.parametrize("n,k", synth.W4A16_ASYM_SHAPES)
def test_full_size_w4a16_asym_sweep(Q, n, k):
    c = Case(max(synth.W4A16_ASYM_MS), n, k, 128, "bf16", False, seed=synth.SEED_W4A16_ASYM)
    lin = linear(c)
    x = c.dev_act()
    ref = c.reference()
    for m in synth.W4A16_ASYM_MS:
        out = lin(x[:m])
        assert lin.status() == Q.QGEMM_OK
        assert_close(to_np(out), ref[:m], what=f"M={m} N={n} K={k}")


def test_full_size_large_every_row(Q):
    """8192^3 INT4 bf16, every one of the 67M outputs against the oracle
    (about 1.1 TFLOP of float64 on the host)."""
    s = synth.LARGE_SHAPE
    c = Case(s["m"], s["n"], s["k"], s["group"], "bf16", True, seed=synth.SEED_LARGE)
    lin = linear(c)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    got = to_np(out)
    del out
    assert_close(got, c.reference(), what="8192^3 every row")


def test_timeout_path_reports_and_recovers(Q):
    c = Case(40, 256, 1024, 128, "bf16", True, seed=3)
    lin = linear(c)
    x = c.dev_act()
    Q.qgemm_set_wait_limit_ns(0)
    try:
        lin(x)
        st = lin.status()
    finally:
        Q.qgemm_set_wait_limit_ns(1_000_000_000)
    assert st == Q.QGEMM_ERR_TIMEOUT
    lin.ws.buf.zero_()              # counters may be left mid-count after an abandoned launch
    out = lin(x)
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what="after timeout")


def test_error_paths_launch_nothing(Q):
    c = Case(8, 256, 256, 128, "bf16", True)
    lin = linear(c)
    x = c.dev_act()
    out = torch.empty(8, 256, dtype=torch.bfloat16, device=DEV)
    st, need = Q.qgemm_workspace_size(lin.layer, lin.dense, None, 8)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    run = lambda **kw: Q.qgemm_run(kw.get("layer", lin.layer), kw.get("compute", lin.dense), None,
                                   kw.get("m", 8), kw.get("a", x), None, lin.packed, None,
                                   kw.get("c", out), kw.get("ws", ws), kw.get("wsb", need))
    assert run(wsb=need - 1) == Q.QGEMM_ERR_WORKSPACE
    assert run(a=x.data_ptr() + 2) == Q.QGEMM_ERR_INVALID_ARG
    assert run(c=0) == Q.QGEMM_ERR_INVALID_ARG
    assert run(m=-1) == Q.QGEMM_ERR_INVALID_ARG
    assert run(compute=lin.grouped) == Q.QGEMM_ERR_INVALID_ARG
    bad = Q.layer_config(200, 256, 128, Q.QGEMM_W_INT4_SYM, Q.QGEMM_S_BF16, Q.QGEMM_Z_NONE,
                         Q.QGEMM_BF16, Q.QGEMM_BF16)
    assert run(layer=bad) == Q.QGEMM_ERR_UNSUPPORTED
    assert "multiples of 128" in Q.last_error()
    torch.cuda.synchronize()
    assert lin.status() == Q.QGEMM_OK


def test_describe_plan_records_choice(Q):
    c = Case(8, 256, 256, 128, "bf16", False)
    lin = linear(c)
    st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, 16)
    assert st == Q.QGEMM_OK and "block_tok=16" in rec and "uint4_zp" in rec
    st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, 1024)
    assert "block_tok=128" in rec


def test_grouped_gemm_parity_with_empty_and_ragged_experts(Q):
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    e, n, k, g = 5, 256, 384, 128
    r = synth.rng(41)
    cases = [Case(1, n, k, g, "bf16", True, seed=100 + i) for i in range(e)]
    rows = [7, 0, 40, 1, 19]
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    total = int(offsets[-1])
    a = codecs.bf16(synth.activations_fp32(r, total, k))
    qw = torch.from_numpy(np.concatenate([cs.qweight for cs in cases])).to(DEV)
    sc = torch.from_numpy(np.concatenate([cs.s_bits for cs in cases]).view(np.int16)).to(DEV)
    lin = W4A16Linear(qw, sc, None, n, k, g, torch.bfloat16, num_experts=e)
    out = lin.run_grouped(torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(DEV),
                          torch.from_numpy(offsets).to(DEV))
    assert lin.status() == Q.QGEMM_OK
    got = to_np(out)
    for i in range(e):
        r0, r1 = offsets[i], offsets[i + 1]
        if r1 > r0:
            assert_close(got[r0:r1], a[r0:r1] @ cases[i].w_hat, what=f"expert {i}")
