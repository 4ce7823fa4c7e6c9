"""GEMM references and the per-token FP8 and NVFP4 activation quantizers.

The Humming pages describe the kernels' work as a GEMM over quantized weights
assembled from scheduling, data movement, dequantization and scaling, tensor
core compute and output processing (kinachrichten.com, "Kompilierzeiten und
gerätespezifisches Tuning"), for W4A16 and for W4A8-MXFP4 (same article, the
MXFP4 paragraph; jetabc.cn post, "跑得有多快", items 1-4).  Readings taken:

W4A16:  C = A @ W^ with W^ the dequantized weights already rounded once to the
        activation dtype (the weights are fed to 16-bit tensor cores), the
        product formed exactly in float64, an optional per-column bias added
        before the single final rounding to the output dtype (= the
        activation dtype).

W4A8:   per token m:  s_m = fp32(max_k |x_mk|) / 448 in fp32 (s_m = 1 if the
        row is all zero);  a8_mk = e4m3_rne_satfinite(fp32(x_mk) / s_m) with
        an IEEE fp32 divide.  Then
            C[m, n] = s_m * sum_b 2^(E_bn) * sum_{k in b} a8_mk * e2m1(c_nk)
        in float64, rounded once to bf16 (the output dtype of this path).

W4A4:   NVFP4 weights and NVFP4 activations (the pages list W4A4 among the
        common configurations and name NVFP4: kinachrichten.com, "Warum
        quantisierte Kernel wichtig sind").  The pages do not say how the
        activations are quantized; the reading taken is NVFP4's two-level
        scaling with a per-tensor fp32 scale a_ts supplied by the caller and
        an e4m3 scale per 16 consecutive k of each token, decided in fp32
        (``act_quant_nvfp4``).  Then
            C[m, n] = a_ts * w_ts * sum_k A[m, k] W[k, n]
        with A = e2m1(a_codes) * e4m3(a_sb) and W = e2m1(w_codes) * e4m3(w_sb)
        the exact operands, in float64, plus the bias, rounded once to bf16.

Split-K, tiling and accumulation order are the kernels' business and do not
appear here; the tests bound their effect with the stated tolerances.
"""

from __future__ import annotations

import numpy as np

from . import codecs, quant


def matmul_f64(a, b) -> np.ndarray:
    """Exact-input float64 product (a library matmul serves as the step)."""
    return np.asarray(a, dtype=np.float64) @ np.asarray(b, dtype=np.float64)


def w4a16_reference(a, w_hat, bias=None) -> np.ndarray:
    """float64 C = A @ W^ (+ bias), before the output rounding."""
    c = matmul_f64(a, w_hat)
    if bias is not None:
        c = c + np.asarray(bias, dtype=np.float64)[None, :]
    return c


def w4a16_output(a, w_hat, out_dt: str, bias=None) -> np.ndarray:
    """C rounded once to the output dtype (values as float64)."""
    return codecs.round_dtype(out_dt)(w4a16_reference(a, w_hat, bias))


def act_quant_fp8(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-token FP8 quantization of activations x[M, K] (bf16 values).

    Returns (e4m3 codes uint8 [M, K], scales float32 [M]).  The scale and the
    divide are fp32 operations, as the kernel performs them, so that the codes
    (an integer decided by floating point) are taken in the same precision on
    both sides."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    amax = np.max(np.abs(x32), axis=1)
    s = (amax / np.float32(448.0)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    scaled = (x32 / s[:, None]).astype(np.float32)        # IEEE fp32 divide
    codes = codecs.encode_e4m3(scaled.astype(np.float64))
    return codes, s


def w4a8_reference(a8_codes, a_scale, w_codes_kn, w_b) -> np.ndarray:
    """float64 C[m, n] = s_m * sum_b 2^(E_bn) * sum_{k in b} a8 * e2m1(c)."""
    a8 = codecs.decode_e4m3(a8_codes)                     # [M, K]
    wv = codecs.decode_e2m1(w_codes_kn)                   # [K, N]
    k = wv.shape[0]
    nb = k // 32
    acc = np.zeros((a8.shape[0], wv.shape[1]), dtype=np.float64)
    scale = codecs.decode_e8m0(w_b)                       # [K/32, N]
    for b in range(nb):
        part = a8[:, 32 * b: 32 * b + 32] @ wv[32 * b: 32 * b + 32, :]
        acc += part * scale[b][None, :]
    return acc * np.asarray(a_scale, dtype=np.float64)[:, None]


def w4a8_output(a8_codes, a_scale, w_codes_kn, w_b) -> np.ndarray:
    return codecs.bf16(w4a8_reference(a8_codes, a_scale, w_codes_kn, w_b))


def act_quant_nvfp4(x, a_ts) -> tuple[np.ndarray, np.ndarray]:
    """Per-token NVFP4 quantization of activations x[M, K] (bf16 values, K a
    multiple of 16) in blocks of 16 along K, against the tensor scale a_ts.

    Returns (codes uint8 [M, K] e2m1 nibbles, sb uint8 [M, K/16] e4m3 bytes),
    x[m, k] ~ e2m1(codes[m, k]) * e4m3(sb[m, k/16]) * a_ts.  Every step is the
    fp32 operation the kernel performs, so that the codes (integers decided by
    floating point) are taken in the same precision on both sides:
        d = fp32(6 * a_ts);  t = fp32(amax / d)     (amax of the block, exact)
        s = e4m3(t)                                  (RNE, satfinite)
        q = fp32(x / fp32(s * a_ts));  code = e2m1(q)  (RNE, saturating at 6,
                                                      the sign of x kept)
    A block whose s is 0 takes code 0 everywhere."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    m, k = x32.shape
    xb = x32.reshape(m, k // 16, 16)
    amax = np.max(np.abs(xb), axis=2)
    a_ts32 = np.float32(a_ts)
    d = np.float32(np.float32(6.0) * a_ts32)
    t = (amax / d).astype(np.float32)                      # IEEE fp32 divide
    s = codecs.e4m3(t.astype(np.float64))
    sb = codecs.encode_e4m3(s)
    denom = (s.astype(np.float32) * a_ts32).astype(np.float32)
    live = denom > 0
    q = (xb / np.where(live, denom, np.float32(1.0))[:, :, None]).astype(np.float32)
    codes = codecs.encode_e2m1(q.astype(np.float64))
    codes = np.where(live[:, :, None], codes, 0)
    return codes.reshape(m, k).astype(np.uint8), sb.astype(np.uint8)


def nvfp4_act_operand(codes, sb) -> np.ndarray:
    """A[m, k] = e2m1(codes[m, k]) * e4m3(sb[m, k/16]), exact in float64."""
    return codecs.decode_e2m1(codes) * np.repeat(codecs.decode_e4m3(sb), 16, axis=1)


def w4a4_reference(a_codes, a_sb, a_ts, w_codes_kn, w_sb_kn, w_ts, bias=None) -> np.ndarray:
    """float64 C[m, n] = a_ts * w_ts * sum_k A[m, k] W[k, n] (+ bias[n])."""
    acc = matmul_f64(nvfp4_act_operand(a_codes, a_sb), quant.nvfp4_operand(w_codes_kn, w_sb_kn))
    c = acc * (float(a_ts) * float(w_ts))
    if bias is not None:
        c = c + np.asarray(bias, dtype=np.float64)[None, :]
    return c


def w4a4_output(a_codes, a_sb, a_ts, w_codes_kn, w_sb_kn, w_ts, bias=None) -> np.ndarray:
    return codecs.bf16(w4a4_reference(a_codes, a_sb, a_ts, w_codes_kn, w_sb_kn, w_ts, bias))


def check_close(gpu, ref, atol=1e-2, rtol=1e-2, frob=5e-3):
    """Acceptance: |gpu - ref| <= atol + rtol |ref| per element and
    ||gpu - ref||_F / ||ref||_F <= frob.  Returns (ok, max_violation, rel_frob)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    worst = float(np.max(err - bound)) if err.size else -1.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(gpu - ref) / denom) if denom > 0 else float(np.linalg.norm(gpu))
    ok = bool(np.all(err <= bound) and rel <= frob and np.all(np.isfinite(gpu)))
    return ok, worst, rel


def dense_from_standard_int(qweight, scales_bits, qzeros, k, g, sdt, adt, signed):
    """Convenience: standard-format tensors -> W^ (the dequantized weights)."""
    q = quant.unpack_int4_kn(qweight, signed)
    s = codecs.dtype_from_bits(sdt, scales_bits)
    z = None if qzeros is None else quant.unpack_zeros(qzeros)
    return quant.dequant_int(q, s, z, g, adt)
