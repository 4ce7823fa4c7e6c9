"""Torch-facing convenience layer over the C ABI.

PyTorch only provides device memory and streams here: each class allocates
the packed weights and the workspace as torch tensors once and then calls the
library's entry points (``qgemm.py``) on the current torch stream.  No
arithmetic of the method runs in Python.
"""

from __future__ import annotations

import torch

from . import qgemm as Q

_DT = {torch.float16: Q.QGEMM_FP16, torch.bfloat16: Q.QGEMM_BF16}


class Workspace:
    """A zero-initialised device workspace that grows on demand."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


class W4A16Linear:
    """A packed W4A16 layer (dense, or the stacked experts of a grouped layer).

    qweight int32 [E*K/8, N], scales [E*K/g, N] (16-bit: the bits of
    ``scale_dtype``, which defaults to the activation dtype; fp16 scales
    also serve bf16 activations), qzeros int32 [E*K/g, N/8] or None: the
    standard format of ``include/qgemm.h``.  gated=True: the N columns are an
    MoE gate half and up half and the layer writes silu(gate) * up, [rows,
    N/2] (bf16 only).  batch_invariant=True: a row's result does not depend on
    the other rows of a call."""

    def __init__(self, qweight, scales, qzeros, n, k, group, act_dtype, num_experts=1,
                 bias=None, tuning=None, deterministic=False, gated=False,
                 batch_invariant=False, scale_dtype=None):
        self.n, self.k, self.group, self.num_experts = n, k, group, num_experts
        self.gated = gated
        self.n_out = n // 2 if gated else n
        self.act_dtype = act_dtype
        asym = qzeros is not None
        adt = _DT[act_dtype]
        sdt = adt if scale_dtype is None else _DT[scale_dtype]
        self.layer = Q.layer_config(
            n, k, group, Q.QGEMM_W_UINT4_ZP if asym else Q.QGEMM_W_INT4_SYM,
            Q.QGEMM_S_FP16 if sdt == Q.QGEMM_FP16 else Q.QGEMM_S_BF16,
            Q.QGEMM_Z_UINT4 if asym else Q.QGEMM_Z_NONE, adt, adt,
            1 if bias is not None else 0, num_experts,
            Q.QGEMM_ACT_SILU_GLU if gated else Q.QGEMM_ACT_NONE)
        self._pack(qweight, scales, qzeros, bias, tuning, deterministic, batch_invariant)

    def _pack(self, qweight, scales, qzeros, bias, tuning, deterministic, batch_invariant):
        """Packs the standard-format tensors for ``self.layer`` (qzeros: the
        zero points, NVFP4's tensor scales, or None) and sets up the configs."""
        st, nbytes = Q.qgemm_packed_size(self.layer)
        Q.check(st)
        dev = qweight.device
        qweight, scales = qweight.contiguous(), scales.contiguous()
        qzeros = None if qzeros is None else qzeros.contiguous()
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        Q.check(Q.qgemm_pack_weights(self.layer, qweight, scales, qzeros, self.packed))
        self.bias = bias
        self.tuning = tuning
        self.ws = Workspace(dev)
        det = 1 if deterministic else 0
        inv = 1 if batch_invariant else 0
        self.dense = Q.compute_config(Q.QGEMM_GEMM_DENSE, batch_invariant=inv, deterministic=det)
        self.grouped = Q.compute_config(Q.QGEMM_GEMM_GROUPED, batch_invariant=inv,
                                        deterministic=det)

    def __call__(self, a: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
        a = a.contiguous()
        m = a.shape[0]
        if out is None:
            out = torch.empty(m, self.n_out, dtype=self.act_dtype, device=a.device)
        st, nbytes = Q.qgemm_workspace_size(self.layer, self.dense, self.tuning, max(m, 1))
        Q.check(st)
        ws = self.ws.get(nbytes)
        Q.check(Q.qgemm_run(self.layer, self.dense, self.tuning, m, a, None, self.packed,
                            self.bias, out, ws, ws.numel()))
        return out

    def run_grouped(self, a_perm: torch.Tensor, offsets: torch.Tensor,
                    out: torch.Tensor | None = None) -> torch.Tensor:
        rows = a_perm.shape[0]
        if out is None:
            out = torch.empty(rows, self.n_out, dtype=self.act_dtype, device=a_perm.device)
        st, nbytes = Q.qgemm_workspace_size(self.layer, self.grouped, self.tuning, max(rows, 1))
        Q.check(st)
        ws = self.ws.get(nbytes)
        Q.check(Q.qgemm_grouped_run(self.layer, self.grouped, self.tuning, offsets, rows, a_perm,
                                    None, self.packed, self.bias, out, ws, ws.numel()))
        return out

    def dequantized(self) -> torch.Tensor:
        """W^[K, N] as the kernels feed it to the tensor core (expert 0)."""
        out = torch.empty(self.k, self.n, dtype=self.act_dtype, device=self.packed.device)
        Q.check(Q.qgemm_debug_dequant(self.layer, self.packed, out))
        return out

    def status(self) -> int:
        return Q.qgemm_check_status(self.ws.get(256))


class W8A16Linear(W4A16Linear):
    """A packed layer of 8-bit integer weights against fp16/bf16 activations:
    qweight int32 [E*K/4, N] (four codes a word along K; INT8 two's complement,
    or UINT8 with qzeros int32 [E*K/g, N/4]), scales [E*K/g, N] in the
    activation dtype.  Runs, grouped runs and the dequantized view are those
    of ``W4A16Linear``."""

    def __init__(self, qweight, scales, qzeros, n, k, group, act_dtype, num_experts=1,
                 bias=None, tuning=None, deterministic=False, gated=False,
                 batch_invariant=False):
        self.n, self.k, self.group, self.num_experts = n, k, group, num_experts
        self.gated = gated
        self.n_out = n // 2 if gated else n
        self.act_dtype = act_dtype
        asym = qzeros is not None
        adt = _DT[act_dtype]
        self.layer = Q.layer_config(
            n, k, group, Q.QGEMM_W_UINT8_ZP if asym else Q.QGEMM_W_INT8_SYM,
            Q.QGEMM_S_FP16 if adt == Q.QGEMM_FP16 else Q.QGEMM_S_BF16,
            Q.QGEMM_Z_UINT8 if asym else Q.QGEMM_Z_NONE, adt, adt,
            1 if bias is not None else 0, num_experts,
            Q.QGEMM_ACT_SILU_GLU if gated else Q.QGEMM_ACT_NONE)
        self._pack(qweight, scales, qzeros, bias, tuning, deterministic, batch_invariant)


class W3A16Linear(W4A16Linear):
    """A packed layer of 3-bit integer weights (GPTQ INT3, or UINT3 with zero
    points) against fp16/bf16 activations: qweight int32 [E*3K/32, N] (each
    column's codes a bit stream along K), scales [E*K/g, N] (16-bit:
    ``scale_dtype``, default the activation dtype), qzeros int32
    [E*K/g, 3N/32] or None.  The pack stores the codes in the 4-bit blocks,
    so runs, grouped runs and the dequantized view are those of
    ``W4A16Linear``."""

    def __init__(self, qweight, scales, qzeros, n, k, group, act_dtype, num_experts=1,
                 bias=None, tuning=None, deterministic=False, gated=False,
                 batch_invariant=False, scale_dtype=None):
        self.n, self.k, self.group, self.num_experts = n, k, group, num_experts
        self.gated = gated
        self.n_out = n // 2 if gated else n
        self.act_dtype = act_dtype
        asym = qzeros is not None
        adt = _DT[act_dtype]
        sdt = adt if scale_dtype is None else _DT[scale_dtype]
        self.layer = Q.layer_config(
            n, k, group, Q.QGEMM_W_UINT3_ZP if asym else Q.QGEMM_W_INT3_SYM,
            Q.QGEMM_S_FP16 if sdt == Q.QGEMM_FP16 else Q.QGEMM_S_BF16,
            Q.QGEMM_Z_UINT3 if asym else Q.QGEMM_Z_NONE, adt, adt,
            1 if bias is not None else 0, num_experts,
            Q.QGEMM_ACT_SILU_GLU if gated else Q.QGEMM_ACT_NONE)
        self._pack(qweight, scales, qzeros, bias, tuning, deterministic, batch_invariant)


class NVFP4Linear(W4A16Linear):
    """A packed layer of NVFP4 weights against fp16/bf16 activations: e2m1
    codes uint8 [E*N, K/2] (standard nibble order), e4m3 block scales uint8
    [E*N, K/16] and fp32 tensor scales [E].  Runs, grouped runs and the
    dequantized view are those of ``W4A16Linear``."""

    def __init__(self, codes, scales, tensor_scales, n, k, act_dtype, num_experts=1, bias=None,
                 tuning=None, deterministic=False, gated=False, batch_invariant=False):
        self.n, self.k, self.group, self.num_experts = n, k, 16, num_experts
        self.gated = gated
        self.n_out = n // 2 if gated else n
        self.act_dtype = act_dtype
        adt = _DT[act_dtype]
        self.layer = Q.layer_config(
            n, k, 16, Q.QGEMM_W_NVFP4, Q.QGEMM_S_E4M3, Q.QGEMM_Z_NONE, adt, adt,
            1 if bias is not None else 0, num_experts,
            Q.QGEMM_ACT_SILU_GLU if gated else Q.QGEMM_ACT_NONE)
        self._pack(codes, scales, tensor_scales.to(torch.float32), bias, tuning, deterministic,
                   batch_invariant)


class W4A8Linear:
    """A packed W4A8-MXFP4 layer: e2m1 codes uint8 [E*N, K/2] and e8m0 scales
    uint8 [E*N, K/32] in the standard format; activations are quantized per
    row to e4m3 by the library and the output is bf16 (gated=True: as for
    W4A16Linear, silu(gate) * up of the two column halves, [rows, N/2]).
    Calling the layer on bf16 activations is one library call (the layer
    config with bf16 activations: the quantization runs inside the small-M
    kernel, or as its own kernel ahead of the tcgen05 one); ``quantize`` and
    ``run_quantized`` are the two-call form with caller-held e4m3 codes."""

    def __init__(self, codes, scales, n, k, num_experts=1, bias=None, tuning=None,
                 deterministic=False, gated=False, batch_invariant=False):
        self.n, self.k, self.num_experts = n, k, num_experts
        self.gated = gated
        self.n_out = n // 2 if gated else n
        cfg = (n, k, 32, Q.QGEMM_W_MXFP4, Q.QGEMM_S_E8M0, Q.QGEMM_Z_NONE)
        tail = (Q.QGEMM_BF16, 1 if bias is not None else 0, num_experts,
                Q.QGEMM_ACT_SILU_GLU if gated else Q.QGEMM_ACT_NONE)
        self.layer = Q.layer_config(*cfg, Q.QGEMM_FP8E4M3, *tail)      # e4m3 activations
        self.layer_bf16 = Q.layer_config(*cfg, Q.QGEMM_BF16, *tail)    # library-quantized
        st, nbytes = Q.qgemm_packed_size(self.layer)
        Q.check(st)
        dev = codes.device
        codes, scales = codes.contiguous(), scales.contiguous()
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        Q.check(Q.qgemm_pack_weights(self.layer, codes, scales, None, self.packed))
        self.bias, self.tuning = bias, tuning
        self.ws = Workspace(dev)
        det = 1 if deterministic else 0
        inv = 1 if batch_invariant else 0
        self.dense = Q.compute_config(Q.QGEMM_GEMM_DENSE, batch_invariant=inv, deterministic=det)
        self.grouped = Q.compute_config(Q.QGEMM_GEMM_GROUPED, batch_invariant=inv,
                                        deterministic=det)
        self._act = {}

    def quantize(self, x: torch.Tensor):
        """x bf16 [M, K] -> (e4m3 codes uint8 [M, K], fp32 scales [M])."""
        m = x.shape[0]
        a8 = torch.empty(m, self.k, dtype=torch.uint8, device=x.device)
        sc = torch.empty(max(m, 1), dtype=torch.float32, device=x.device)
        Q.check(Q.qgemm_quantize_act_fp8(x, m, self.k, a8, sc))
        return a8, sc

    def run_quantized(self, a8, a_scale, out=None):
        m = a8.shape[0]
        if out is None:
            out = torch.empty(m, self.n_out, dtype=torch.bfloat16, device=a8.device)
        st, nbytes = Q.qgemm_workspace_size(self.layer, self.dense, self.tuning, max(m, 1))
        Q.check(st)
        ws = self.ws.get(nbytes)
        Q.check(Q.qgemm_run(self.layer, self.dense, self.tuning, m, a8, a_scale, self.packed,
                            self.bias, out, ws, ws.numel()))
        return out

    def __call__(self, x: torch.Tensor, out=None) -> torch.Tensor:
        """x bf16 [M, K] -> bf16 [M, N] in one library call."""
        x = x.contiguous()
        m = x.shape[0]
        if out is None:
            out = torch.empty(m, self.n_out, dtype=torch.bfloat16, device=x.device)
        st, nbytes = Q.qgemm_workspace_size(self.layer_bf16, self.dense, self.tuning, max(m, 1))
        Q.check(st)
        ws = self.ws.get(nbytes)
        Q.check(Q.qgemm_run(self.layer_bf16, self.dense, self.tuning, m, x, None, self.packed,
                            self.bias, out, ws, ws.numel()))
        return out

    def two_call(self, x: torch.Tensor, out=None) -> torch.Tensor:
        """The same product through qgemm_quantize_act_fp8, then qgemm_run."""
        a8, sc = self.quantize(x.contiguous())
        return self.run_quantized(a8, sc, out)

    def codes_e4m3(self) -> torch.Tensor:
        """The e4m3 bytes the kernel feeds the tensor core, uint8 [K, N]."""
        out = torch.empty(self.k, self.n, dtype=torch.uint8, device=self.packed.device)
        Q.check(Q.qgemm_debug_dequant(self.layer, self.packed, out))
        return out

    def status(self) -> int:
        return Q.qgemm_check_status(self.ws.get(256))


class W4A4Linear:
    """A packed W4A4 layer: NVFP4 weights (e2m1 codes uint8 [N, K/2] in the
    standard nibble order, e4m3 block scales uint8 [N, K/16], one fp32 tensor
    scale) against activations the library quantizes to NVFP4 per token
    against ``act_scale`` (a device fp32 [1] tensor scale).  Calling the layer
    on bf16 activations is one library call (the quantization kernel, then the
    FP4 tensor-core GEMM); ``quantize`` exposes the quantization alone."""

    def __init__(self, codes, scales, tensor_scale, act_scale, n, k, bias=None, tuning=None):
        self.n, self.k, self.n_out = n, k, n
        self.layer = Q.layer_config(n, k, 16, Q.QGEMM_W_NVFP4, Q.QGEMM_S_E4M3, Q.QGEMM_Z_NONE,
                                    Q.QGEMM_NVFP4, Q.QGEMM_BF16, 1 if bias is not None else 0, 1,
                                    Q.QGEMM_ACT_NONE)
        st, nbytes = Q.qgemm_packed_size(self.layer)
        Q.check(st)
        dev = codes.device
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        ts = tensor_scale.to(torch.float32).reshape(-1)[:1].contiguous()
        Q.check(Q.qgemm_pack_weights(self.layer, codes.contiguous(), scales.contiguous(), ts,
                                     self.packed))
        self.act_scale = act_scale.to(torch.float32).reshape(-1)[:1].contiguous()
        self.bias, self.tuning = bias, tuning
        self.ws = Workspace(dev)
        self.dense = Q.compute_config(Q.QGEMM_GEMM_DENSE)

    def quantize(self, x: torch.Tensor):
        """x bf16 [M, K] -> (e2m1 codes uint8 [M, K/2], e4m3 block scales uint8 [M, K/16])."""
        m = x.shape[0]
        codes = torch.empty(max(m, 1), self.k // 2, dtype=torch.uint8, device=x.device)
        sb = torch.empty(max(m, 1), self.k // 16, dtype=torch.uint8, device=x.device)
        Q.check(Q.qgemm_quantize_act_nvfp4(x.contiguous(), m, self.k, self.act_scale, codes, sb))
        return codes[:m], sb[:m]

    def __call__(self, x: torch.Tensor, out=None) -> torch.Tensor:
        """x bf16 [M, K] -> bf16 [M, N]."""
        x = x.contiguous()
        m = x.shape[0]
        if out is None:
            out = torch.empty(m, self.n, dtype=torch.bfloat16, device=x.device)
        st, nbytes = Q.qgemm_workspace_size(self.layer, self.dense, self.tuning, max(m, 1))
        Q.check(st)
        ws = self.ws.get(nbytes)
        Q.check(Q.qgemm_run(self.layer, self.dense, self.tuning, m, x, self.act_scale,
                            self.packed, self.bias, out, ws, ws.numel()))
        return out

    def status(self) -> int:
        return Q.qgemm_check_status(self.ws.get(256))


class MoELayer:
    """Grouped-MoE W4A16 layer: permute -> GEMM1 (gate|up) -> SiLU gate ->
    GEMM2 (down) -> combine, all on the current stream, no host sync.  When
    w1 is gated the SiLU gate runs in GEMM1's epilogue (one launch fewer,
    no [rows, 2I] intermediate)."""

    def __init__(self, w1: W4A16Linear, w2: W4A16Linear, num_experts: int, topk: int):
        self.w1, self.w2 = w1, w2
        self.e, self.topk = num_experts, topk
        self.hidden = w1.k
        self.inter = w2.k
        self._bufs = {}

    def buffers(self, t: int, device):
        if t not in self._bufs:
            r = t * self.topk
            bf = torch.bfloat16
            self._bufs[t] = dict(
                offsets=torch.empty(self.e + 1, dtype=torch.int32, device=device),
                perm=torch.empty(max(r, 1), dtype=torch.int32, device=device),
                inv=torch.empty(max(r, 1), dtype=torch.int32, device=device),
                a_perm=torch.empty(max(r, 1), self.hidden, dtype=bf, device=device),
                gu=(None if self.w1.gated else
                    torch.empty(max(r, 1), 2 * self.inter, dtype=bf, device=device)),
                h=torch.empty(max(r, 1), self.inter, dtype=bf, device=device),
                y2=torch.empty(max(r, 1), self.hidden, dtype=bf, device=device),
            )
        return self._bufs[t]

    def __call__(self, a, topk_ids, topk_weights, out=None, keep=False):
        t = a.shape[0]
        b = self.buffers(t, a.device)
        r = t * self.topk
        if out is None:
            out = torch.empty(t, self.hidden, dtype=torch.bfloat16, device=a.device)
        Q.check(Q.qgemm_moe_permute(topk_ids, t, self.topk, self.e, b["offsets"], b["perm"],
                                    b["inv"], a, b["a_perm"], self.hidden))
        if self.w1.gated:
            self.w1.run_grouped(b["a_perm"][:r], b["offsets"], out=b["h"][:r])
        else:
            self.w1.run_grouped(b["a_perm"][:r], b["offsets"], out=b["gu"][:r])
            Q.check(Q.qgemm_moe_silu_mul(b["gu"], r, self.inter, b["h"]))
        self.w2.run_grouped(b["h"][:r], b["offsets"], out=b["y2"][:r])
        Q.check(Q.qgemm_moe_combine(b["y2"], b["inv"], topk_weights, t, self.topk, self.hidden,
                                    out))
        if keep:
            return out, b
        return out
