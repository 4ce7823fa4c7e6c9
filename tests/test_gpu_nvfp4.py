"""GPU parity of NVFP4 weights (e2m1 codes, an e4m3 scale per 16 k, an fp32
tensor scale per expert) against fp16/bf16 activations, through the C ABI:
the pack and the values fed to the tensor core bit for bit, the GEMM within
|gpu - ref| <= 1e-2 + 1e-2 |ref| per element and relative Frobenius error
<= 5e-3, dense, split-K, grouped and gated."""

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import DEV, TD, assert_close, to_np
from oracle import codecs, gemm, layout, moe, quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from quantized_weight_gemm_run_b300 import qgemm
    qgemm.qgemm_set_wait_limit_ns(1_000_000_000)
    return qgemm


class NvCase:
    """E experts of NVFP4 weights [K, N] quantized by the oracle, and rows."""

    def __init__(self, m, n, k, adt, seed, experts=1, bias=False):
        g = synth.rng(seed)
        self.m, self.n, self.k, self.adt, self.e = m, n, k, adt, experts
        self.codes, self.sb, self.t, self.w_hat = [], [], [], []
        for _ in range(experts):
            w = synth.weights_fp32(g, k, n)
            c, sb, t = quant.quantize_nvfp4(w)
            self.codes.append(c)
            self.sb.append(sb)
            self.t.append(t)
            self.w_hat.append(quant.dequant_nvfp4(c, sb, t))
        self.a = codecs.round_dtype(adt)(synth.activations_fp32(g, m, k))
        self.bias = codecs.round_dtype(adt)(g.standard_normal(n) * 0.5) if bias else None

    def standard(self):
        packed = [quant.pack_nvfp4(c, s) for c, s in zip(self.codes, self.sb)]
        codes = np.concatenate([p[0] for p in packed])
        sb = np.concatenate([p[1] for p in packed])
        return codes, sb

    def layer(self, **kw):
        from quantized_weight_gemm_run_b300.api import NVFP4Linear
        codes, sb = self.standard()
        bias = None
        if self.bias is not None:
            bias = torch.from_numpy(self.bias.astype(np.float32)).to(TD[self.adt]).to(DEV)
        return NVFP4Linear(torch.from_numpy(codes).to(DEV), torch.from_numpy(sb).to(DEV),
                           torch.tensor(self.t, dtype=torch.float32, device=DEV), self.n, self.k,
                           TD[self.adt], num_experts=self.e, bias=bias, **kw)

    def a_dev(self, rows=None):
        a = self.a if rows is None else self.a[rows]
        return torch.from_numpy(a.astype(np.float32)).to(TD[self.adt]).to(DEV)

    def reference(self, e=0, rows=None):
        a = self.a if rows is None else self.a[rows]
        return gemm.w4a16_reference(a, self.w_hat[e], self.bias)


@pytest.mark.parametrize("adt,experts,gated", [("bf16", 1, False), ("fp16", 1, False),
                                               ("bf16", 3, False), ("bf16", 1, True)])
def test_nvfp4_pack_bit_exact(Q, adt, experts, gated):
    c = NvCase(4, 384, 512, adt, seed=71 + experts, experts=experts)
    lin = c.layer(gated=gated)
    torch.cuda.synchronize()
    il = layout.glu_interleave_columns if gated else (lambda x, axis=-1: x)
    want = []
    for i in range(experts):
        cn, sn = quant.pack_nvfp4(c.codes[i], c.sb[i])
        want.append(layout.packed_nvfp4(il(cn, axis=0), il(sn, axis=0), adt))
    want = np.concatenate(want + [layout.nvfp4_tail(c.t)])
    assert np.array_equal(lin.packed.cpu().numpy(), want)


@pytest.mark.parametrize("adt", ["bf16", "fp16"])
def test_nvfp4_operand_bit_exact(Q, adt):
    c = NvCase(4, 256, 384, adt, seed=73)
    lin = c.layer()
    deq = lin.dequantized().cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, codecs.dtype_bits(adt, quant.nvfp4_operand(c.codes[0], c.sb[0])))


def test_nvfp4_all_codes_and_scales(Q):
    """Every e2m1 code in every nibble position against every e4m3 scale byte."""
    from quantized_weight_gemm_run_b300.api import NVFP4Linear
    k, n = 128 * 16, 128
    codes = np.tile(np.arange(16, dtype=np.uint8), (k * n) // 16).reshape(k, n)
    codes = np.roll(codes, 5, axis=1)
    sb = (np.arange((k // 16) * n) % 0x7F).astype(np.uint8).reshape(k // 16, n)
    cn, sn = quant.pack_nvfp4(codes, sb)
    for adt in ("bf16", "fp16"):
        lin = NVFP4Linear(torch.from_numpy(cn).to(DEV), torch.from_numpy(sn).to(DEV),
                          torch.ones(1, dtype=torch.float32, device=DEV), n, k, TD[adt])
        deq = lin.dequantized().cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(deq, codecs.dtype_bits(adt, quant.nvfp4_operand(codes, sb))), adt


SMALL = [
    # m, n, k, adt, bias
    (1, 128, 128, "bf16", False),
    (16, 256, 256, "fp16", False),
    (37, 384, 512, "bf16", True),
    (130, 256, 1024, "fp16", True),
    (300, 640, 384, "bf16", False),
]


@pytest.mark.parametrize("m,n,k,adt,bias", SMALL)
def test_nvfp4_gemm_small_parity(Q, m, n, k, adt, bias):
    c = NvCase(m, n, k, adt, seed=m + n + k, bias=bias)
    lin = c.layer()
    out = lin(c.a_dev())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"nvfp4 {m}x{n}x{k} {adt}")


@pytest.mark.parametrize("bt", [16, 128])
@pytest.mark.parametrize("det", [False, True])
def test_nvfp4_split_tiles(Q, bt, det):
    c = NvCase(45, 384, 2048, "bf16", seed=75)
    lin = c.layer(tuning=Q.tuning_config(block_tok=bt, max_ctas=7), deterministic=det)
    out = lin(c.a_dev())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what=f"nvfp4 split bt={bt} det={det}")


def test_nvfp4_grouped_ragged_experts(Q):
    """Each expert has its own tensor scale; empty and sub-chunk experts."""
    c = NvCase(0, 256, 512, "bf16", seed=76, experts=5)
    rows = [7, 0, 40, 1, 19]
    offsets = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    total = int(offsets[-1])
    a = codecs.bf16(synth.activations_fp32(synth.rng(77), total, c.k))
    lin = c.layer()
    out = lin.run_grouped(torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(DEV),
                          torch.from_numpy(offsets).to(DEV))
    assert lin.status() == Q.QGEMM_OK
    got = to_np(out)
    for i in range(c.e):
        r0, r1 = offsets[i], offsets[i + 1]
        if r1 > r0:
            assert_close(got[r0:r1], a[r0:r1] @ c.w_hat[i], what=f"expert {i}")


def test_nvfp4_gated(Q):
    c = NvCase(37, 384, 512, "bf16", seed=78)
    lin = c.layer(gated=True)
    out = lin(c.a_dev())
    assert out.shape == (37, 192) and lin.status() == Q.QGEMM_OK
    ref = moe.silu_mul(codecs.bf16(c.reference()), 192)
    assert_close(to_np(out), ref, what="nvfp4 gated")


def test_nvfp4_full_size_m256(Q):
    """M = 256, N = K = 4096 (a sweep shape), every element against the oracle."""
    c = NvCase(256, 4096, 4096, "bf16", seed=79)
    lin = c.layer()
    out = lin(c.a_dev())
    assert lin.status() == Q.QGEMM_OK
    assert_close(to_np(out), c.reference(), what="nvfp4 256x4096x4096")


def test_nvfp4_m_zero_and_missing_tensor_scales(Q):
    c = NvCase(4, 128, 128, "bf16", seed=80)
    lin = c.layer()
    out = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    assert Q.qgemm_run(lin.layer, lin.dense, None, 0, c.a_dev(), None, lin.packed, None, out,
                       lin.ws.get(256), 256) == Q.QGEMM_OK
    codes, sb = c.standard()
    packed = torch.empty_like(lin.packed)
    assert Q.qgemm_pack_weights(lin.layer, torch.from_numpy(codes).to(DEV),
                                torch.from_numpy(sb).to(DEV), None, packed) == \
        Q.QGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("adt", ["bf16", "fp16"])
def test_small_m_kernel_operands_every_code_and_scale(Q, adt):
    """The small-M kernel's own NVFP4 path (m <= 16): one-hot activation rows
    pick single weight rows, so each output is one operand times the tensor
    scale 2^-3 (exact, as are the fp32 sums of zeros).  16 calls of 16 rows
    cover one row of every 16-k block: every code in every nibble position
    against every e4m3 scale byte, compared with the oracle's operand."""
    from quantized_weight_gemm_run_b300.api import NVFP4Linear
    k, n = 128 * 16, 128
    codes = np.tile(np.arange(16, dtype=np.uint8), (k * n) // 16).reshape(k, n)
    codes = np.roll(codes, 5, axis=1)
    sb = (np.arange((k // 16) * n) % 0x7F).astype(np.uint8).reshape(k // 16, n)
    cn, sn = quant.pack_nvfp4(codes, sb)
    ts = 0.125
    lin = NVFP4Linear(torch.from_numpy(cn).to(DEV), torch.from_numpy(sn).to(DEV),
                      torch.full((1,), ts, dtype=torch.float32, device=DEV), n, k, TD[adt],
                      tuning=Q.tuning_config(kernel=2))
    st, rec = Q.qgemm_describe_plan(lin.layer, lin.dense, 16)
    assert "kernel=w4a16_mma_sync_smallm" in rec, rec
    want = quant.nvfp4_operand(codes, sb) * ts
    blocks = k // 16
    for call in range(blocks // 16):
        rows = [(call * 16 + i) * 16 + (call * 5 + 3 * i) % 16 for i in range(16)]
        x = np.zeros((16, k), dtype=np.float32)
        x[np.arange(16), rows] = 1.0
        out = lin(torch.from_numpy(x).to(TD[adt]).to(DEV))
        assert lin.status() == Q.QGEMM_OK
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.array_equal(got, codecs.round_dtype(adt)(want[rows])), f"{adt} call {call}"


@pytest.mark.parametrize("m", [1, 9, 16])
def test_small_m_kernel_matches_oracle_and_tcgen05(Q, m):
    c = NvCase(m, 384, 1024, "bf16", seed=200 + m, bias=True)
    small = c.layer(tuning=Q.tuning_config(kernel=2))
    big = c.layer(tuning=Q.tuning_config(kernel=1))
    x = c.a_dev()
    o2 = small(x)
    o1 = big(x)
    assert small.status() == Q.QGEMM_OK and big.status() == Q.QGEMM_OK
    ref = c.reference()
    assert_close(to_np(o2), ref, what=f"nvfp4 small-M m={m}")
    assert_close(to_np(o1), ref, what=f"nvfp4 tcgen05 m={m}")


def test_plan_routes_nvfp4_by_layer_size(Q):
    """The small-M kernel takes NVFP4 layers of up to 2^24 weights at m <= 16,
    and larger ones at m <= 8 when K <= 4096; the rest go to the tcgen05 kernel."""
    import copy
    lin = NvCase(4, 256, 256, "bf16", seed=231).layer()
    for m, n, k, kern in ((16, 4096, 4096, "w4a16_mma_sync_smallm"),
                          (8, 11008, 4096, "w4a16_mma_sync_smallm"),
                          (9, 11008, 4096, "w4a16_tcgen05_swapab"),
                          (1, 4096, 11008, "w4a16_tcgen05_swapab"),
                          (17, 4096, 4096, "w4a16_tcgen05_swapab")):
        cfg = copy.copy(lin.layer)
        cfg.n, cfg.k = n, k
        st, rec = Q.qgemm_describe_plan(cfg, lin.dense, m)
        assert st == Q.QGEMM_OK
        assert f"kernel={kern}" in rec, (m, n, k, rec)
