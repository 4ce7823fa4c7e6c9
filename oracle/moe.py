"""Grouped-MoE reference: routing, permutation, expert GEMMs, SiLU gate, combine.

The pages motivate the MoE path by tokens activating only a subset of experts
while all expert weights stay resident (kinachrichten.com, "Warum quantisierte
Kernel wichtig sind") and report a grouped-MoE path on B300 (jetabc.cn post,
"跑得有多快", item 3).  The layer itself is not specified on the pages;
readings taken:

  routing  : probabilities p = softmax(logits) per token (float64); the top-k
             experts by probability, ties to the lower expert index; the
             routing weights are those k probabilities, NOT renormalised,
             handed to both sides as float32.
  permute  : flat slots i = t * k + j sorted stably by expert id, giving
             expert_offsets[E + 1] and perm[T * k] (perm[r] = slot at row r);
             A_perm[r] = A[perm[r] // k].
  GEMM1    : GU = adt(A_perm[rows of e] @ W1^_e), W1 columns = [gate | up].
  act      : H = bf16(silu(G) * U), silu in float64 of the bf16 inputs.
  GEMM2    : Y2 = bf16(H[rows of e] @ W2^_e).
  combine  : Y[t] = bf16(sum_j w[t, j] * Y2[pos(t, j)]), pos = inverse perm,
             summed in float64 in the order j = 0 .. k-1.
"""

from __future__ import annotations

import numpy as np

from . import codecs


def route(logits, topk: int):
    """-> (topk_ids int32 [T, k], topk_weights float32 [T, k])."""
    lg = np.asarray(logits, dtype=np.float64)
    mx = lg.max(axis=1, keepdims=True)
    ex = np.exp(lg - mx)
    p = ex / ex.sum(axis=1, keepdims=True)
    t, e = p.shape
    ids = np.empty((t, topk), dtype=np.int32)
    wts = np.empty((t, topk), dtype=np.float32)
    for i in range(t):
        order = sorted(range(e), key=lambda x: (-p[i, x], x))[:topk]
        ids[i] = order
        wts[i] = p[i, order].astype(np.float32)
    return ids, wts


def permute(topk_ids, num_experts: int):
    """Stable counting sort of the T*k slots by expert.

    -> (expert_offsets int32 [E+1], perm int32 [T*k])."""
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    counts = np.bincount(ids, minlength=num_experts)
    offsets = np.zeros(num_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(ids, kind="stable")
    return offsets.astype(np.int32), perm.astype(np.int32)


def gather_rows(a, perm, topk: int):
    return np.asarray(a)[np.asarray(perm) // topk]


def silu_mul(gu, inter: int) -> np.ndarray:
    """H = bf16(silu(G) * U) for GU = [G | U] (bf16 values, float64 math)."""
    gu = np.asarray(gu, dtype=np.float64)
    g = gu[:, :inter]
    u = gu[:, inter:2 * inter]
    silu = g / (1.0 + np.exp(-g))
    return codecs.bf16(silu * u)


def grouped_gemm(x, offsets, w_hat_fn, out_dt: str) -> np.ndarray:
    """Rows [offsets[e], offsets[e+1]) of x times W^_e, rounded to out_dt.

    ``w_hat_fn(e)`` returns expert e's dequantized weights [K, N] (float64)."""
    x = np.asarray(x, dtype=np.float64)
    out = None
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        w = w_hat_fn(e)
        if out is None:
            out = np.zeros((x.shape[0], w.shape[1]), dtype=np.float64)
        out[r0:r1] = x[r0:r1] @ w
    if out is None:
        out = np.zeros((x.shape[0], 0))
    return codecs.round_dtype(out_dt)(out)


def combine(y2, perm, topk_weights, topk: int) -> np.ndarray:
    """Y[t] = bf16(sum_j w[t, j] * Y2[pos(t, j)])."""
    y2 = np.asarray(y2, dtype=np.float64)
    perm = np.asarray(perm, dtype=np.int64)
    w = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    t = w.shape[0]
    pos = np.empty_like(perm)
    pos[perm] = np.arange(perm.size)
    acc = np.zeros((t, y2.shape[1]), dtype=np.float64)
    for j in range(topk):
        acc += w[:, j][:, None] * y2[pos.reshape(t, topk)[:, j]]
    return codecs.bf16(acc)


def moe_layer(a, topk_ids, topk_weights, w1_hat_fn, w2_hat_fn, num_experts, inter, adt="bf16"):
    """The whole layer; returns a dict of every intermediate (float64 values)."""
    topk = topk_ids.shape[1]
    offsets, perm = permute(topk_ids, num_experts)
    a_perm = gather_rows(a, perm, topk)
    gu = grouped_gemm(a_perm, offsets, w1_hat_fn, adt)
    h = silu_mul(gu, inter)
    y2 = grouped_gemm(h, offsets, w2_hat_fn, "bf16")
    y = combine(y2, perm, topk_weights, topk)
    return dict(offsets=offsets, perm=perm, a_perm=a_perm, gu=gu, h=h, y2=y2, y=y)
