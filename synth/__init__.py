"""Seeded synthetic inputs for the quantized-weight GEMM workloads.

This module is the only code shared between the CPU oracle and the CUDA path's
tests and benchmark.  It draws random numbers and random bit patterns and holds
none of the method's arithmetic: no quantization, no packing, no rounding to a
narrow format, no GEMM.  Everything it returns is either float32 data (weights,
activations, router logits) or uniformly random raw words/bytes that stand in
for already-quantized tensors when only their size and layout matter (timing).

Workload recipe (the five workload families of the Humming announcement's
kernel microbenchmarks, restated with explicit sizes):

  * W4A16 dense, symmetric INT4, fp16:   M=16, N=K=4096, group 128, seed 0
  * W4A16 dense, asymmetric UINT4, bf16: (N,K) in {(4096,4096), (11008,4096),
    (4096,11008)} x M in {1,4,16,64,256,1024}, group 128, seed 1
  * W4A8-MXFP4: N=7168, K=2048, M in {1,8,32,128,512}, seed 2
  * grouped MoE W4A16: E=64, top-8, hidden 2048, intermediate 1408,
    T in {16,256,4096}, seed 3
  * large-batch W4A16: M=N=K=8192, bf16, symmetric INT4 group 128, seed 4

Weights are drawn as fp32 ~ N(0, 0.02) and laid out [K, N] (row k, column n);
activations as fp32 ~ N(0, 1) laid out [M, K]; router logits fp32 ~ N(0, 1)
laid out [T, E].  Generation order inside one workload: weights, then
activations, then logits, all from one numpy Generator seeded as above.
"""

from __future__ import annotations

import numpy as np

WEIGHT_STD = 0.02
ACT_STD = 1.0

SEED_W4A16_SYM = 0
SEED_W4A16_ASYM = 1
SEED_W4A8 = 2
SEED_MOE = 3
SEED_LARGE = 4

W4A16_SYM_SHAPE = dict(m=16, n=4096, k=4096, group=128)
W4A16_ASYM_SHAPES = [(4096, 4096), (11008, 4096), (4096, 11008)]
W4A16_ASYM_MS = [1, 4, 16, 64, 256, 1024]
W4A8_SHAPE = dict(n=7168, k=2048)
W4A8_MS = [1, 8, 32, 128, 512]
MOE_SHAPE = dict(experts=64, topk=8, hidden=2048, inter=1408, group=128)
MOE_TS = [16, 256, 4096]
LARGE_SHAPE = dict(m=8192, n=8192, k=8192, group=128)


def rng(seed: int) -> np.random.Generator:
    """One numpy PCG64 generator per workload, seeded as documented above."""
    return np.random.default_rng(seed)


def weights_fp32(g: np.random.Generator, k: int, n: int, std: float = WEIGHT_STD) -> np.ndarray:
    """Dense fp32 weights laid out [K, N], ~N(0, std)."""
    return g.standard_normal((k, n), dtype=np.float32) * np.float32(std)


def expert_weights_fp32(g: np.random.Generator, e: int, k: int, n: int,
                        std: float = WEIGHT_STD) -> np.ndarray:
    """Stacked per-expert fp32 weights laid out [E, K, N], ~N(0, std)."""
    return g.standard_normal((e, k, n), dtype=np.float32) * np.float32(std)


def activations_fp32(g: np.random.Generator, m: int, k: int, std: float = ACT_STD) -> np.ndarray:
    """Dense fp32 activations laid out [M, K], ~N(0, std)."""
    return g.standard_normal((m, k), dtype=np.float32) * np.float32(std)


def router_logits_fp32(g: np.random.Generator, t: int, e: int) -> np.ndarray:
    """Router logits laid out [T, E], ~N(0, 1)."""
    return g.standard_normal((t, e), dtype=np.float32)


def random_words(g: np.random.Generator, shape, dtype=np.int32) -> np.ndarray:
    """Uniformly random raw words (every bit pattern equally likely).

    Stands in for packed 4-bit codes when only the tensor's size matters."""
    info = np.iinfo(dtype)
    return g.integers(info.min, info.max, size=shape, dtype=dtype, endpoint=True)


def random_scales_fp32(g: np.random.Generator, shape, lo: float = 0.004,
                       hi: float = 0.012) -> np.ndarray:
    """Positive fp32 scale magnitudes, uniform in [lo, hi).

    The default range brackets the absmax/7 (or range/15) scales that
    N(0, 0.02) weights in groups of 128 produce."""
    return g.uniform(lo, hi, size=shape).astype(np.float32)


def random_bytes(g: np.random.Generator, shape, lo: int = 0, hi: int = 255) -> np.ndarray:
    """Uniform random bytes in [lo, hi] (inclusive)."""
    return g.integers(lo, hi, size=shape, dtype=np.uint8, endpoint=True)
