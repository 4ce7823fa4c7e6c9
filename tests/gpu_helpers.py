"""Shared helpers of the GPU parity tests: build a case with the oracle, run it
through the library's C ABI, compare."""

from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import codecs, gemm, quant

TD = {"bf16": torch.bfloat16, "fp16": torch.float16}
DEV = "cuda"


class Case:
    """One W4A16 problem, quantized by the oracle from seeded fp32 data."""

    def __init__(self, m, n, k, g, adt, sym, seed=0, bias=False, sdt=None):
        r = synth.rng(seed)
        w = synth.weights_fp32(r, k, n)
        sdt = adt if sdt is None else sdt             # the scale dtype
        self.a = codecs.round_dtype(adt)(synth.activations_fp32(r, m, k))
        if sym:
            self.q, self.s = quant.quantize_int4_sym(w, g, sdt)
            self.z = None
        else:
            self.q, self.s, self.z = quant.quantize_uint4_asym(w, g, sdt)
        self.m, self.n, self.k, self.g, self.adt, self.sym = m, n, k, g, adt, sym
        self.sdt = sdt
        self.qweight = quant.pack_int4_kn(self.q, sym)
        self.s_bits = codecs.dtype_bits(sdt, self.s)
        self.qzeros = None if self.z is None else quant.pack_zeros(self.z)
        self.w_hat = quant.dequant_int(self.q, self.s, self.z, g, adt)
        self.bias = codecs.round_dtype(adt)(r.standard_normal(n) * 0.5) if bias else None

    def dev_weights(self):
        qw = torch.from_numpy(self.qweight).to(DEV)
        sc = torch.from_numpy(self.s_bits.view(np.int16)).to(DEV)
        qz = None if self.qzeros is None else torch.from_numpy(self.qzeros).to(DEV)
        return qw, sc, qz

    def dev_act(self):
        return torch.from_numpy(self.a.astype(np.float32)).to(TD[self.adt]).to(DEV)

    def dev_bias(self):
        if self.bias is None:
            return None
        return torch.from_numpy(self.bias.astype(np.float32)).to(TD[self.adt]).to(DEV)

    def reference(self, rows=None):
        a = self.a if rows is None else self.a[rows]
        return gemm.w4a16_reference(a, self.w_hat, self.bias)


def linear(case: Case, tuning=None, deterministic=False):
    from quantized_weight_gemm_run_b300.api import W4A16Linear
    qw, sc, qz = case.dev_weights()
    return W4A16Linear(qw, sc, qz, case.n, case.k, case.g, TD[case.adt], bias=case.dev_bias(),
                       tuning=tuning, deterministic=deterministic, scale_dtype=TD[case.sdt])


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(gpu, ref, frob=5e-3, what=""):
    ok, worst, rel = gemm.check_close(gpu, ref, frob=frob)
    assert ok, f"{what}: worst excess {worst:.3g}, relative Frobenius {rel:.3g}"
    return rel
