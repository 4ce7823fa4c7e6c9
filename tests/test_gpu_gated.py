"""GPU parity of the SiLU-gated output (an MoE expert's gate|up projection
with the gate applied in the GEMM's epilogue), through the C ABI: the gated
pack bit for bit against the oracle's layout, the fused output against the
oracle's GEMM followed by its SiLU gate within the GEMM tolerance, and bit for
bit against the library's own unfused path (GEMM, then the SiLU kernel) when
both run the same whole-tile schedule."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import DEV, TD, Case, assert_close, to_np
from oracle import codecs, gemm, layout, moe, quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


def _lin(c: Case, gated, tuning=None, deterministic=False):
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    qw, sc, qz = c.dev_weights()
    return W4A16Linear(qw, sc, qz, c.n, c.k, c.g, TD[c.adt], bias=c.dev_bias(), tuning=tuning,
                       deterministic=deterministic, gated=gated)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _gated_ref(c: Case, rows=None):
    return moe.silu_mul(codecs.bf16(c.reference(rows)), c.n // 2)


@pytest.mark.parametrize("sym,g", [(True, 128), (False, 32), (False, 256)])
def test_gated_pack_bit_exact_and_dequant_in_standard_order(Q, sym, g):
    c = Case(4, 384, 512, g, "bf16", sym, seed=61)
    lin = _lin(c, gated=True)
    torch.cuda.synchronize()
    il = layout.glu_interleave_columns
    want = layout.packed_w4(il(c.q), il(c.s_bits), None if c.z is None else il(c.z), g,
                            signed=sym)
    assert np.array_equal(lin.packed.cpu().numpy(), want)
    assert np.array_equal(_bits(lin.dequantized()), codecs.dtype_bits("bf16", c.w_hat))


GATED = [
    # m, n, k, g, sym, bias
    (1, 128, 128, 128, True, False),
    (16, 256, 256, 128, False, False),
    (37, 384, 512, 128, True, True),
    (70, 640, 768, 64, False, False),
    (129, 256, 1024, 128, True, False),
    (300, 512, 384, 32, False, True),
]


@pytest.mark.parametrize("m,n,k,g,sym,bias", GATED)
def test_gated_gemm_parity(Q, m, n, k, g, sym, bias):
    c = Case(m, n, k, g, "bf16", sym, seed=m + n + k + 1, bias=bias)
    lin = _lin(c, gated=True)
    out = lin(c.dev_act())
    assert out.shape == (m, n // 2)
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), _gated_ref(c), what=f"gated {m}x{n}x{k}")


@pytest.mark.parametrize("bt", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("det,max_ctas", [(False, 7), (True, 7), (False, 0)])
def test_gated_split_tiles(Q, bt, det, max_ctas):
    """Split-K tiles (few CTAs, many k-tiles) reach the gated output through
    the finisher and the fixed-order sum as well."""
    c = Case(45, 384, 2048, 128, "bf16", False, seed=77)
    lin = _lin(c, gated=True, tuning=Q.tuning_config(block_tok=bt, max_ctas=max_ctas),
               deterministic=det)
    out = lin(c.dev_act())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), _gated_ref(c), what=f"gated split bt={bt} det={det}")


@pytest.mark.parametrize("m,bt", [(37, 16), (200, 64), (300, 128)])
def test_gated_equals_unfused_bits(Q, m, bt):
    """With whole tiles only (no split-K), each output column's fp32 sum is
    the same in both layouts, so the fused epilogue must give exactly the bits
    of the GEMM followed by the standalone SiLU kernel."""
    c = Case(m, 512, 1024, 128, "bf16", True, seed=m + 3, bias=True)
    tun = Q.tuning_config(block_tok=bt, split_k=1)
    fused = _lin(c, gated=True, tuning=tun)(c.dev_act())
    gu = _lin(c, gated=False, tuning=tun)(c.dev_act())
    h = torch.empty(m, c.n // 2, dtype=torch.bfloat16, device=DEV)
    Q.check(Q.qgemm_moe_silu_mul(gu, m, c.n // 2, h))
    assert torch.equal(fused.view(torch.int16), h.view(torch.int16))


def test_gated_grouped_ragged_experts(Q):
    """Grouped gated GEMM: empty experts, experts smaller than a chunk (the
    row-by-row stores of a tile's last chunk) and several tiles."""
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    e, n, k, g = 5, 384, 512, 128
    r = synth.rng(42)
    cases = [Case(1, n, k, g, "bf16", False, seed=200 + i) for i in range(e)]
    rows = [7, 0, 40, 1, 19]
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    total = int(offsets[-1])
    a = codecs.bf16(synth.activations_fp32(r, total, k))
    qw = torch.from_numpy(np.concatenate([cs.qweight for cs in cases])).to(DEV)
    sc = torch.from_numpy(np.concatenate([cs.s_bits for cs in cases]).view(np.int16)).to(DEV)
    qz = torch.from_numpy(np.concatenate([cs.qzeros for cs in cases])).to(DEV)
    a_dev = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(DEV)
    off_dev = torch.from_numpy(offsets).to(DEV)
    for bt in (16, 64):
        lin = W4A16Linear(qw, sc, qz, n, k, g, torch.bfloat16, num_experts=e, gated=True,
                          tuning=Q.tuning_config(block_tok=bt))
        out = lin.run_grouped(a_dev, off_dev)
        assert out.shape == (total, n // 2)
        assert lin.status() == Q.QGEMM_OK
        got = to_np(out)
        for i in range(e):
            r0, r1 = offsets[i], offsets[i + 1]
            if r1 > r0:
                ref = moe.silu_mul(codecs.bf16(a[r0:r1] @ cases[i].w_hat), n // 2)
                assert_close(got[r0:r1], ref, what=f"bt={bt} expert {i}")


def test_gated_w4a8_parity_and_pack(Q):
    from quantized_weight_gemm_run_b300.api import W4A8Linear
    m, n, k = 37, 384, 512
    g = synth.rng(63)
    w = synth.weights_fp32(g, k, n)
    x = codecs.bf16(synth.activations_fp32(g, m, k))
    codes_kn, b_kn = quant.quantize_mxfp4(w)
    codes_nk, b_nk = quant.pack_mxfp4(codes_kn, b_kn)
    lin = W4A8Linear(torch.from_numpy(codes_nk).to(DEV), torch.from_numpy(b_nk).to(DEV), n, k,
                     gated=True)
    torch.cuda.synchronize()
    il = layout.glu_interleave_columns
    want = layout.packed_mxfp4(il(codes_nk, axis=0), il(b_nk, axis=0))
    assert np.array_equal(lin.packed.cpu().numpy(), want)
    assert np.array_equal(lin.codes_e4m3().cpu().numpy(),
                          codecs.encode_e4m3(codecs.decode_e2m1(codes_kn)))
    out = lin(torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(DEV))
    assert lin.status() == Q.QGEMM_OK
    a8, s = gemm.act_quant_fp8(x)
    ref = moe.silu_mul(codecs.bf16(gemm.w4a8_reference(a8, s, codes_kn, b_kn)), n // 2)
    assert_close(to_np(out), ref, frob=2e-2, what="gated w4a8")


def test_gated_rejects_fp16(Q):
    c = Case(4, 256, 256, 128, "fp16", True)
    with pytest.raises(Q.QGemmError):
        _lin(c, gated=True)
