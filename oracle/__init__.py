"""CPU oracle for the quantized-weight GEMM hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the library path imports, calls or links
anything here; only the tests, the smoke check in ``__graft_entry__`` and the
CPU-baseline leg of ``bench.py`` may use it.  It shares no code with the CUDA
path: its formats, layouts and arithmetic are written out here from their
definitions, in plain NumPy, in float64 unless a step fixes another precision.

What it computes follows the Humming pages (the jetabc.cn post "一个库吃下所有量化
格式：蚂蚁和 vLLM 开源推理内核库 Humming" and the kinachrichten.com article "Ant
Group und vLLM stellen Humming als Open Source vor"): a quantized weight is a
tensor of low-bit codes plus group scales and optional zero points (the
"standard format"), which a preprocessing step checks and repacks for a kernel,
and which a GEMM consumes as weights against 16-bit or 8-bit activations,
dense or grouped over MoE experts.  The pages print no formulas; the readings
taken where they are silent are stated in each function's docstring.

Modules:
  codecs  -- bf16 / fp16 / e4m3 / e2m1 / e8m0 encode and decode
  quant   -- quantizers, the standard-format packing, dequantization
  layout  -- the kernel-side packed layout the repack step must produce
  gemm    -- W4A16, W4A8 and W4A4 GEMM references, per-token FP8 and NVFP4
             activation quantizers
  moe     -- routing, permutation, SiLU-gate, combine, the full MoE layer

Parity status: every function is pinned by tests under ``tests/`` (tables,
closed forms, brute force, invariants).  The throughput figures the pages
quote have no per-shape numbers and are "parity unpinned" by nature: they are
reported as context only.
"""

from . import codecs, quant, layout, gemm, moe  # noqa: F401
