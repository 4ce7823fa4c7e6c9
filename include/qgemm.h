/*
 * qgemm.h -- C ABI of the B300 (sm_103a) quantized-weight GEMM library.
 *
 * The library runs the hot path of a mixed-precision GEMM over quantized
 * weights: W4A16 (INT4 / UINT4 codes with per-group fp16 or bf16 scales and
 * optional zero points, dequantized in registers and fed to 16-bit tensor-core
 * MMA with fp32 accumulation; also NVFP4 codes, and 8-bit INT8 / UINT8 codes
 * as W8A16), W4A8-MXFP4 (e2m1 codes with e8m0 per-32 scales against per-token
 * FP8 e4m3 activations) and the grouped-MoE variant that runs one such GEMM
 * per expert over router-permuted tokens.
 *
 * Where the operations come from (the Humming pages; titles and sections):
 *   - kinachrichten.com, "Ant Group und vLLM stellen Humming als Open Source
 *     vor: Kernel-Bibliothek fuer quantisierte Inferenz", section "Wie die
 *     Architektur funktioniert": a standard format for weights, scales, zero
 *     points; a preprocessing step that checks parameters, pads and repacks
 *     for the target kernel; three configurations per kernel (Layer, Compute,
 *     Tuning); device heuristics choosing the tuning, with different kernels
 *     for different input-size ranges.  Section "Kompilierzeiten und
 *     geraetespezifisches Tuning": kernels built from scheduling, data
 *     movement, dequantization/scaling, tensor-core compute and output
 *     processing components; the W4A8-MXFP4 path.
 *   - jetabc.cn, "一个库吃下所有量化格式：蚂蚁和 vLLM 开源推理内核库 Humming",
 *     section "Humming 的做法" (standard format, three configs) and
 *     "跑得有多快" (W4A16, grouped MoE and W4A8-MXFP4 kernel families).
 *   - retrivium.ai retrospective "vLLM Humming: why shared quantization still
 *     needs specialized kernels", section "The architectural gain is a smaller
 *     maintenance surface": unsupported combinations are rejected clearly.
 *
 * Conventions for every entry point:
 *   - All tensors are caller-owned.  Pointers marked "device" are CUDA device
 *     pointers on the current device; the library allocates no device memory
 *     and never frees caller memory.  Pointers must be 16-byte aligned; every
 *     tensor is dense row-major with the strides implied by its shape.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous on it and never synchronize, except qgemm_check_status.
 *   - Arguments are validated synchronously on the host; on any error nothing
 *     is launched and a status != QGEMM_OK is returned.  qgemm_last_error()
 *     returns a human-readable reason for the last failing call of the thread.
 *   - Unsupported combinations (e.g. zero points with MXFP4, N or K not a
 *     multiple of 128, K not a multiple of the group size) return
 *     QGEMM_ERR_UNSUPPORTED.  There is no fallback path.
 *   - A CUDA launch error returns QGEMM_ERR_CUDA.
 */
#ifndef QGEMM_H_
#define QGEMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QGEMM_OK = 0,
  QGEMM_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment        */
  QGEMM_ERR_UNSUPPORTED = 2, /* valid but not implemented combination       */
  QGEMM_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required  */
  QGEMM_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed           */
  QGEMM_ERR_TIMEOUT = 5,     /* a kernel gave up a bounded wait             */
  QGEMM_ERR_DEVICE = 6       /* a kernel reported an internal error         */
} qgemm_status;

/* weight formats */
enum {
  QGEMM_W_INT4_SYM = 0,
  QGEMM_W_UINT4_ZP = 1,
  QGEMM_W_MXFP4 = 2,
  QGEMM_W_NVFP4 = 3,
  QGEMM_W_INT8_SYM = 4,   /* W8A16 */
  QGEMM_W_UINT8_ZP = 5,
  QGEMM_W_INT3_SYM = 6,   /* GPTQ INT3 (W3A16) */
  QGEMM_W_UINT3_ZP = 7
};
/* scale formats */
enum { QGEMM_S_FP16 = 0, QGEMM_S_BF16 = 1, QGEMM_S_E8M0 = 2, QGEMM_S_E4M3 = 3 };
/* zero-point formats */
enum { QGEMM_Z_NONE = 0, QGEMM_Z_UINT4 = 1, QGEMM_Z_UINT8 = 2, QGEMM_Z_UINT3 = 3 };
/* activation / output data types */
enum { QGEMM_FP16 = 0, QGEMM_BF16 = 1, QGEMM_FP8E4M3 = 2, QGEMM_NVFP4 = 3 };
/* GEMM types (compute config) */
enum { QGEMM_GEMM_DENSE = 0, QGEMM_GEMM_GROUPED = 1 };
/* gated activation fused into the output (layer config) */
enum { QGEMM_ACT_NONE = 0, QGEMM_ACT_SILU_GLU = 1 };

/*
 * Layer config: what the layer is.  Shapes are those of one expert; a dense
 * layer has num_experts = 1.
 *   n, k          output features, input features (C[M,N] = A[M,K] W[K,N])
 *   group_size    K-extent of one scale (W4A16 and W8A16: 32, 64 or a
 *                 multiple of 128 dividing K; MXFP4: must be 32; NVFP4: must
 *                 be 16)
 *   weight_format QGEMM_W_*;  scale_format QGEMM_S_*;  zero_format QGEMM_Z_*
 *   act_dtype     activation dtype: QGEMM_FP16 / QGEMM_BF16 (W4A16, W8A16
 *                 with 8-bit integer weights and scales in the activation
 *                 dtype: the pages list weight-only formats WNA16,
 *                 kinachrichten.com "Warum quantisierte Kernel wichtig
 *                 sind", and
 *                 NVFP4 weights: e2m1 codes, one e4m3 scale per 16 k, one
 *                 fp32 tensor scale; the pages name NVFP4 as a format whose
 *                 number format and scaling differ from INT4's,
 *                 kinachrichten.com "Warum quantisierte Kernel wichtig sind") or
 *                 QGEMM_FP8E4M3 (W4A8; the caller passes e4m3 codes and
 *                 per-row fp32 scales from qgemm_quantize_act_fp8) or
 *                 QGEMM_BF16 with MXFP4 weights (W4A8 whose bf16 activations
 *                 the library quantizes with the qgemm_quantize_act_fp8 rule:
 *                 at m <= 8 inside the small-M kernel, above in a separate
 *                 kernel into the workspace; results are bitwise those of the
 *                 two-call form; such a layer's workspace then holds its
 *                 quantized rows, so it must not be shared with other layers)
 *                 or QGEMM_NVFP4 with NVFP4 weights (W4A4: the pages list
 *                 W4A4 among the common configurations, kinachrichten.com
 *                 "Warum quantisierte Kernel wichtig sind"; the caller passes
 *                 bf16 activations and, as a_scale, one fp32 activation
 *                 tensor scale on the device, and the library quantizes each
 *                 token to e2m1 codes with an e4m3 scale per 16 k by the
 *                 qgemm_quantize_act_nvfp4 rule into the workspace, then runs
 *                 both operands packed through the FP4 tensor cores; dense,
 *                 ungated, k a multiple of 256, bf16 output; the workspace
 *                 holds the quantized rows and must not be shared)
 *   out_dtype     output dtype: equal to act_dtype for W4A16, QGEMM_BF16 for W4A8
 *                 and W4A4
 *   has_bias      1: add bias[N] (out_dtype) in fp32 before the final rounding
 *   num_experts   1 for a dense layer, E for a grouped (MoE) layer
 *   gated_act     QGEMM_ACT_NONE: C[M, N] = A W (+ bias).
 *                 QGEMM_ACT_SILU_GLU: the N columns of W are a gate half G
 *                 (columns [0, N/2)) and an up half U (columns [N/2, N)) of
 *                 an expert's first MoE projection; the output is
 *                 H[M, N/2] = silu(G') * U', where G' and U' are the two
 *                 halves of A W (+ bias) rounded to out_dtype, silu in fp32,
 *                 the product rounded to out_dtype (bit-identical to running
 *                 the layer with QGEMM_ACT_NONE and then qgemm_moe_silu_mul).
 *                 The weights are passed in the standard format and order;
 *                 the pack entry point interleaves the two halves so that a
 *                 gate column and its up column land in one output tile.
 *                 Needs out_dtype QGEMM_BF16.
 */
typedef struct {
  int64_t n;
  int64_t k;
  int32_t group_size;
  int32_t weight_format;
  int32_t scale_format;
  int32_t zero_format;
  int32_t act_dtype;
  int32_t out_dtype;
  int32_t has_bias;
  int32_t num_experts;
  int32_t gated_act;
} qgemm_layer_config;

/*
 * Compute config: what computation (GEMM type and options such as batch
 * invariance: kinachrichten.com, "Wie die Architektur funktioniert").
 *   gemm_type       QGEMM_GEMM_DENSE or QGEMM_GEMM_GROUPED
 *   batch_invariant 0: the heuristic may split a tile's K range across CTAs,
 *                   at boundaries that depend on the problem's tile count and
 *                   so on m (or, grouped, on the rows of every expert).
 *                   1: no tile is split (each output is one CTA's sum over
 *                   k-tiles 0, 1, ... in order), so a row's result is
 *                   bitwise the same whatever the other rows of the call are
 *                   and whatever m is.  Slower at small m, where split-K is
 *                   what fills the GPU.
 *   deterministic   0: when a tile's K range is split across CTAs, the fp32
 *                   partial sums are added into an L2-resident accumulator by
 *                   atomic reductions (fastest; the order of those fp32
 *                   additions, and so the last bit of a result, can differ
 *                   between runs).  1: the partial sums are added in a fixed
 *                   CTA order (bitwise reproducible for a given problem,
 *                   tuning and device).
 */
typedef struct {
  int32_t gemm_type;
  int32_t batch_invariant;
  int32_t deterministic;
} qgemm_compute_config;

/*
 * Tuning config: how to run it on this device.  Pass NULL for the built-in
 * B300 heuristic (token tile chosen by the M range).  Fields left 0 are chosen
 * by the heuristic.
 *   block_tok  tokens per tile (the MMA N extent): 16, 32, 64, 128 or 256
 *              (256: INT4 / UINT4 weights with scales in the activation
 *              dtype only; one accumulator buffer)
 *   stages     shared-memory pipeline depth (2 .. 16)
 *   max_ctas   upper bound on the persistent grid (<= number of SMs)
 *   split_k    0 = the heuristic's choice (without max_ctas: whole tiles,
 *              stream-K or, for a dense GEMM, the cluster split, by a cost
 *              model of each; with max_ctas: stream-K); s = 1..64:
 *              the tiles left over after the whole waves are each split
 *              across min(s, grid / tiles left) CTAs at k-tile boundaries
 *              (1 = never split a tile's K range)
 *   cta_pair   reserved, must be 0
 *   kernel     0 = the heuristic's choice, 1 = the tcgen05 kernel,
 *              2 = the small-M kernel (bulk-copied weights, mma.sync, K
 *              slices reduced inside a thread-block cluster; dense INT4 /
 *              UINT4 / INT3 / UINT3 with scales in the activation dtype or
 *              fp16 scales against bf16 activations, NVFP4 weights, and
 *              W4A8-MXFP4, m <= 16 only, not gated or batch-invariant;
 *              split_k, when set, is its number of K slices per n-tile, a
 *              power of two <= 16; stages its weight slots; it ignores the
 *              other fields),
 *              3 = the tcgen05 kernel with the cluster split (dense, not
 *              batch-invariant, block_tok <= 128, max_ctas 0): each output
 *              tile's K range in split_k slices (2..8, <= K/128; 0 = the
 *              heuristic's count), one CTA each, the slices of a tile summed
 *              in a fixed order through distributed shared memory, so the
 *              bits repeat from call to call
 * W4A4 layers (act_dtype QGEMM_NVFP4) take block_tok (16, 32, 64 or 128),
 * split_k and kernel = 1 only: split_k = s (1 .. min(64, K/256)) cuts every
 * tile's K range into s slices, one work item each, whose fp32 partials the
 * last slice to finish sums in slice order (1 = whole tiles; 0 = the
 * heuristic: slices only while the tiles leave SMs idle at small M).
 */
typedef struct {
  int32_t block_tok;
  int32_t stages;
  int32_t max_ctas;
  int32_t split_k;
  int32_t cta_pair;
  int32_t kernel;
} qgemm_tuning_config;

/*
 * Standard-format input tensors (what qgemm_pack_weights consumes).  Weights
 * are the logical matrix W[k, n].  Per expert (stacked on a leading E axis):
 *   INT4 / UINT4:
 *     qweight  int32 [K/8, N]: word (j, n) holds k = 8j + i in bits [4i, 4i+4),
 *              least significant nibble first; INT4 as 4-bit two's complement,
 *              UINT4 as raw 0..15
 *     scales   fp16 or bf16 [K/g, N], row-major (group-major); fp16 scales
 *              serve fp16 or bf16 activations, bf16 scales bf16 activations
 *              (the pages count the representation of the scales among the
 *              axes along which formats vary: kinachrichten.com, "Warum
 *              quantisierte Kernel wichtig sind")
 *     qzeros   int32 [K/g, N/8] (UINT4_ZP only): nibble i of word (G, j) is the
 *              zero point (0..15) of column 8j + i; the stored value is the
 *              true zero point
 *     meaning  w[k, n] = (q - z) * s, rounded once to the activation dtype
 *              (z = 0 for INT4; an fp16 scale with bf16 activations is not
 *              rounded to bf16 first)
 *   INT3 / UINT3 (GPTQ 3-bit codes, W3A16):
 *     qweight  int32 [3K/32, N]: the codes of column n form a little-endian
 *              bit stream along K, code k in bits [3k, 3k+3) of the column's
 *              stream (word 3j + w of the column holds stream bits
 *              [32 (3j + w), 32 (3j + w) + 32)), so 32 codes fill three words
 *              and a code may straddle two; INT3 as 3-bit two's complement
 *              (-4..3), UINT3 as raw 0..7
 *     scales   as INT4
 *     qzeros   int32 [K/g, 3N/32] (UINT3_ZP only): each group row's zero
 *              points as a bit stream along N, column c in bits [3c, 3c+3)
 *     meaning  as INT4.  The pages name GPTQ INT3 among the formats served
 *              (jetabc.cn, "怎么使用").  The pack repacks the codes into the
 *              4-bit blocks (INT3 as offset binary q + 8, UINT3 and its zero
 *              points unchanged), so every 4-bit kernel runs them.
 *   INT8 / UINT8 (W8A16):
 *     qweight  int32 [K/4, N]: word (j, n) holds k = 4j + i in bits [8i, 8i+8),
 *              INT8 as two's complement, UINT8 as raw 0..255
 *     scales   as INT4, in the activation dtype
 *     qzeros   int32 [K/g, N/4] (UINT8_ZP only): byte i of word (G, j) is the
 *              zero point (0..255) of column 4j + i
 *     meaning  as INT4
 *   MXFP4:
 *     codes    uint8 [N, K/2]: byte (n, j) holds k = 2j (low nibble) and
 *              k = 2j + 1 (high nibble) as e2m1 (sign | 2 exponent | 1 mantissa)
 *     scales   uint8 e8m0 [N, K/32]: the block scale 2^(b - 127); 255 is invalid
 *     meaning  w[k, n] = e2m1(code) * 2^(b - 127)
 *   NVFP4:
 *     codes    as MXFP4
 *     scales   uint8 e4m3 [N, K/16]: one block scale per 16 k (NaN codes
 *              0x7F / 0xFF are invalid)
 *     tensor   fp32 [E]: one scale per expert, passed in the qzeros argument
 *     meaning  w[k, n] = e2m1(code) * e4m3(scale) * tensor
 *   NVFP4 for W4A4 (act_dtype QGEMM_NVFP4): the same tensors (E = 1); the
 *     packed buffer is codes [N, K/2], then scales [N, K/16], then the
 *     tensor scale, end to end (the FP4 tensor cores read them as they are)
 */

/*
 * Bytes of the packed (kernel-layout) buffer of one layer (all experts).
 * Returns INVALID_ARG / UNSUPPORTED on a bad config.
 * Source: the preprocessing step that checks the parameters and repacks the
 * tensors for the target kernel (kinachrichten.com, "Wie die Architektur
 * funktioniert"); the buffer's size is that of the repacked tensors.
 */
qgemm_status qgemm_packed_size(const qgemm_layer_config* layer, size_t* bytes);

/*
 * Source: the standard format that every export is converted into
 * (jetabc.cn, "Humming 的做法", item 1) and the preprocessing that checks
 * the parameters and repacks the tensors for the target kernel
 * (kinachrichten.com, "Wie die Architektur funktioniert"); repacking changes
 * the arrangement, never the meaning of the values (retrivium.ai, "vLLM
 * Humming: why shared quantization still needs specialized kernels",
 * section "Representation answers a different question"); preparation is
 * kept apart from repeated execution (retrivium.ai, "humming-format-kernel-
 * contract-release", section "Compilation and measurement boundaries").
 *
 * Preprocessing (the "repack for the target kernel" step): validates the
 * config and rearranges the standard-format tensors (device, layout above)
 * into one packed device buffer (`packed`, qgemm_packed_size bytes, 16-byte
 * aligned).  Per expert, the buffer holds one block per (128-row n-tile,
 * 128-deep k-tile), n-tile major: the tile's codes, then its scales, then its
 * zero points, so that consecutive k-tiles of a tile are contiguous.  INT4
 * and INT8 codes are re-encoded as offset binary (q + 8, q + 128) and NVFP4
 * block scales as the
 * activation dtype's bit pattern of the same value; nothing changes value, so
 * the packed buffer means exactly what the standard tensors mean.  NVFP4
 * buffers end with the fp32 tensor scales (16-byte padded).  qzeros must be
 * NULL unless zero_format is QGEMM_Z_UINT4 or QGEMM_Z_UINT8 (zero points) or the weights are
 * NVFP4 (the tensor scales, required).  Runs once per layer; the
 * buffer is read-only afterwards.  For a gated layer (gated_act != 0) row
 * 2i + s of n-tile nt holds the standard column s * N/2 + 64 nt + i (gate
 * columns on even rows, the matching up columns on odd rows).
 */
qgemm_status qgemm_pack_weights(const qgemm_layer_config* layer, const void* qweight,
                                const void* scales, const void* qzeros, void* packed,
                                void* stream);

/*
 * Workspace bytes qgemm_run / qgemm_grouped_run need for `m` rows (for the
 * grouped call: the total number of permuted rows).  The workspace holds a
 * status word, split-K tile counters and fp32 partial tiles.  It must be
 * zero-filled once before first use (qgemm_workspace_init); every successful
 * call leaves the counters at zero again.  One workspace must not be used by
 * two calls that can run at the same time.
 * Source: its size follows the plan that the device heuristic picks from the
 * tuning config (tile shapes, pipeline stages) for the input-size range, and
 * the scheduling component that splits the K range of a tile across CTAs
 * (kinachrichten.com, "Wie die Architektur funktioniert" and "Kompilierzeiten
 * und geraetespezifisches Tuning").  The caller owns the memory: the library
 * allocates none.
 */
qgemm_status qgemm_workspace_size(const qgemm_layer_config* layer,
                                  const qgemm_compute_config* compute,
                                  const qgemm_tuning_config* tuning, int64_t m, size_t* bytes);

/* Zero-fill a workspace on `stream` (asynchronous).  A helper of this
 * library's workspace convention; the pages have no counterpart. */
qgemm_status qgemm_workspace_init(void* workspace, size_t bytes, void* stream);

/*
 * Dense quantized GEMM: C[m, n] = out_dtype(A[m, :] . W[:, n] (+ bias[n])).
 *   m         rows of A and C (0 is allowed and launches nothing)
 *   a         device, [m, K] in act_dtype (e4m3 codes for W4A8 with
 *             act_dtype QGEMM_FP8E4M3)
 *   a_scale   device fp32 [m] per-row activation scales (W4A8 with e4m3
 *             activations); W4A4: device fp32 [1], the activations' tensor
 *             scale (positive and finite); else NULL (also for W4A8 with
 *             bf16 activations)
 *   packed    device packed buffer from qgemm_pack_weights
 *   bias      device [N] in out_dtype, or NULL when has_bias = 0
 *   c         device, [m, N] in out_dtype ([m, N/2] for a gated layer)
 *   workspace device, >= qgemm_workspace_size bytes, zero-initialised once
 * With compute->deterministic = 1 the split-K reduction runs in a fixed order
 * and results are bitwise reproducible for a given (config, m, tuning, device).
 * Source: one kernel described by a layer config (shapes, data types,
 * quantization parameters), a compute config (the GEMM type and options such
 * as batch invariance) and a tuning config chosen by device heuristics, with
 * different kernels for different input-size ranges (kinachrichten.com, "Wie
 * die Architektur funktioniert"), built from scheduling, data movement,
 * dequantization and scaling, tensor-core compute and output processing
 * (same page, "Kompilierzeiten und geraetespezifisches Tuning", which also
 * describes the W4A8-MXFP4 path); the W4A16 and W4A8-MXFP4 kernel families
 * (jetabc.cn, "跑得有多快", items 1, 2 and 4).  Unsupported combinations are
 * rejected with a clear status (retrivium.ai, "vLLM Humming: why shared
 * quantization still needs specialized kernels", section "The architectural
 * gain is a smaller maintenance surface").
 */
qgemm_status qgemm_run(const qgemm_layer_config* layer, const qgemm_compute_config* compute,
                       const qgemm_tuning_config* tuning, int64_t m, const void* a,
                       const float* a_scale, const void* packed, const void* bias, void* c,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * qgemm_run without a workspace argument, for callers that cannot allocate
 * device memory when they run a GEMM (code running under an allocator or
 * memory-pool lock it does not own, plugins inside a host program that owns
 * every device byte, start-up or recovery paths that must not touch the
 * allocator).  The Humming pages have no counterpart to this entry point.
 * It allocates nothing: the split-K scratch is a fixed 32 MiB array inside
 * the library, held on each GPU until the process exits.  Arguments and
 * results are those of qgemm_run (dense GEMMs only).
 *   - The runtime may load the library's device code lazily: the array
 *     becomes resident on a device when the first call made with that device
 *     current looks up its address.  That lookup can fail for lack of device
 *     memory (QGEMM_ERR_CUDA; the next call tries again), so make the first
 *     call on each device early, and before any stream capture.
 *   - All calls share the array and it keeps the last call's contents: calls
 *     that can overlap on the GPU race and must be serialised by the caller.
 *     Each call, after every argument check has passed, zeroes the scratch its
 *     launch uses (status word, split-K counters and accumulators;
 *     cudaMemsetAsync on `stream`) just before the launch; a call that fails a
 *     check queues nothing.
 *   - A problem needing more than 32 MiB of scratch is rejected with
 *     QGEMM_ERR_UNSUPPORTED before anything is launched (qgemm_last_error
 *     names the size).
 *   - A kernel-side timeout is reported by qgemm_noalloc_check_status.
 */
qgemm_status qgemm_run_noalloc(const qgemm_layer_config* layer,
                               const qgemm_compute_config* compute,
                               const qgemm_tuning_config* tuning, int64_t m, const void* a,
                               const float* a_scale, const void* packed, const void* bias,
                               void* c, void* stream);

/*
 * qgemm_check_status for the scratch of qgemm_run_noalloc on the current
 * device: synchronizes `stream`, reads and clears the status word that the
 * last such call's kernel left, and returns QGEMM_OK, QGEMM_ERR_TIMEOUT or
 * QGEMM_ERR_DEVICE.  No workspace needs re-zeroing afterwards (every
 * qgemm_run_noalloc call clears its scratch).  The pages have no counterpart.
 */
qgemm_status qgemm_noalloc_check_status(void* stream);

/*
 * Grouped (MoE) quantized GEMM over router-permuted rows: for each expert e,
 * rows [offsets[e], offsets[e+1]) of A are multiplied by expert e's weights.
 *   expert_offsets device int32 [E+1], non-decreasing, offsets[0] = 0,
 *                  offsets[E] = total_rows (e.g. from qgemm_moe_permute)
 *   total_rows     number of rows of A and C (host value)
 *   packed         packed buffer of all E experts
 *   bias           device [E, N] or NULL
 *   c              device [total_rows, N] ([total_rows, N/2] when gated)
 * The tile schedule is built on the device from expert_offsets: no host
 * synchronization is needed between the permute and the GEMM.
 * Source: MoE models, where each token activates only some experts while all
 * expert weights stay resident (kinachrichten.com, "Warum quantisierte
 * Kernel wichtig sind"); dense and MoE workloads served by one architecture
 * (same page, "Was Humming bietet"); the GEMM type of the compute config
 * (same page, "Wie die Architektur funktioniert"); the grouped-MoE path on
 * B300 (jetabc.cn, "跑得有多快", item 3).
 */
qgemm_status qgemm_grouped_run(const qgemm_layer_config* layer,
                               const qgemm_compute_config* compute,
                               const qgemm_tuning_config* tuning, const int32_t* expert_offsets,
                               int64_t total_rows, const void* a, const float* a_scale,
                               const void* packed, const void* bias, void* c, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * Per-token FP8 activation quantization (W4A8 path):
 *   a_scale[r] = max_k |x[r, k]| / 448 (fp32; 1 for an all-zero row)
 *   a8[r, k]   = e4m3(x[r, k] / a_scale[r]), IEEE fp32 divide, round to
 *                nearest even, saturating at +-448
 *   x device bf16 [m, k]; a8 device uint8 [m, k]; a_scale device fp32 [m].
 *   k must be a multiple of 8 (QGEMM_ERR_UNSUPPORTED otherwise); x must be
 *   16-byte aligned, a8 8-byte aligned, a_scale 4-byte aligned.
 * Source: quantization lowers the precision of activations as well as weights
 * (kinachrichten.com, "Warum quantisierte Kernel wichtig sind"); the
 * W4A8-MXFP4 path with 8-bit activations (same page, "Kompilierzeiten und
 * geraetespezifisches Tuning"; jetabc.cn, "跑得有多快", item 4).  The pages do
 * not define the activation scale: the per-token absmax / 448 rule above is
 * this library's reading.
 */
qgemm_status qgemm_quantize_act_fp8(const void* x, int64_t m, int64_t k, void* a8,
                                    float* a_scale, void* stream);

/*
 * Per-token NVFP4 activation quantization (W4A4 path), in blocks of 16 along
 * k, against the caller's tensor scale a_ts (device fp32 [1], positive and
 * finite); every step is an fp32 operation:
 *   block_scales[r, b] = e4m3(amax_b / (6 a_ts)), amax_b = max |x[r, 16b..16b+15]|,
 *                        round to nearest even, saturating at 448
 *   codes[r, k]        = e2m1(x[r, k] / (s a_ts)), s the block's e4m3 value,
 *                        IEEE fp32 divide, round to nearest even, saturating
 *                        at +-6, the sign of x kept (a block whose s is 0
 *                        takes code 0 throughout)
 *   x device bf16 [m, k]; codes device uint8 [m, k/2] (k = 2j in the low
 *   nibble of byte j, as the standard NVFP4 weight codes); block_scales
 *   device uint8 [m, k/16].  k must be a multiple of 16; x must be 16-byte
 *   aligned, codes 8-byte aligned, a_ts 4-byte aligned.
 * Source: the pages list W4A4 among the common configurations and name NVFP4
 * (kinachrichten.com, "Warum quantisierte Kernel wichtig sind"); they do not
 * say how activations are quantized: NVFP4's two-level scaling with a
 * caller-supplied tensor scale is this library's reading.
 */
qgemm_status qgemm_quantize_act_nvfp4(const void* x, int64_t m, int64_t k, const float* a_ts,
                                      void* codes, void* block_scales, void* stream);

/*
 * MoE permutation: stable counting sort of the t*topk (token, slot) pairs by
 * expert id, then the row gather.
 *   topk_ids    device int32 [t, topk], values in [0, e); e <= 256.  Ids
 *               outside [0, e) are placed after the last expert (rows
 *               offsets[e] .. t*topk - 1) and join no expert GEMM
 *   offsets     device int32 [e+1] (output): rows of expert x are
 *               [offsets[x], offsets[x+1])
 *   perm        device int32 [t*topk] (output): perm[r] = token*topk + j, the
 *               (token, slot) pair placed at row r; pairs of one expert keep
 *               their (token, slot) order
 *   inv_perm    device int32 [t*topk] (output): inv_perm[token*topk + j] = r
 *   a           device [t, hidden] activations (2-byte elements)
 *   a_perm      device [t*topk, hidden] (output): a_perm[r] = a[perm[r] / topk];
 *               it also holds the sort's per-block histograms until the
 *               gather overwrites it, so it must not overlap a or the ids
 * Source: the MoE routing in which each token activates only a subset of the
 * experts (kinachrichten.com, "Warum quantisierte Kernel wichtig sind"),
 * served by the MoE backend (jetabc.cn, "怎么使用") and the grouped-MoE path
 * (jetabc.cn, "跑得有多快", item 3).  The pages do not define the permute:
 * a stable sort by expert is this library's reading.
 */
qgemm_status qgemm_moe_permute(const int32_t* topk_ids, int64_t t, int32_t topk, int32_t e,
                               int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                               const void* a, void* a_perm, int64_t hidden, void* stream);

/*
 * SiLU gate: h[r, i] = bf16(silu(gu[r, i]) * gu[r, inter + i]) in fp32,
 * gu device bf16 [rows, 2*inter], h device bf16 [rows, inter].
 * Source: the output-processing component of a kernel (kinachrichten.com,
 * "Kompilierzeiten und geraetespezifisches Tuning") in the MoE workloads the
 * library serves (same page, "Warum quantisierte Kernel wichtig sind").  The
 * gated activation itself is this library's reading of an MoE expert.
 */
qgemm_status qgemm_moe_silu_mul(const void* gu, int64_t rows, int64_t inter, void* h,
                                void* stream);

/*
 * Combine: y[t, :] = bf16(sum_{j < topk} w[t, j] * y2[inv_perm[t*topk + j], :])
 * in fp32, summed in slot order j = 0..topk-1.
 *   y2 device bf16 [t*topk, hidden]; inv_perm device int32 [t*topk] (from
 *   qgemm_moe_permute); topk_weights device fp32 [t, topk]; y device bf16
 *   [t, hidden].
 * Source: the MoE layer's last step, where each token's expert outputs are
 * merged (kinachrichten.com, "Warum quantisierte Kernel wichtig sind";
 * jetabc.cn, "跑得有多快", item 3).  The weighted sum in slot order is this
 * library's reading.
 */
qgemm_status qgemm_moe_combine(const void* y2, const int32_t* inv_perm,
                               const float* topk_weights, int64_t t, int32_t topk,
                               int64_t hidden, void* y, void* stream);

/*
 * Debug: the weights of a packed layer (expert 0 or the dense layer) as the
 * kernels feed them to the tensor core, written as out[k, n] (device, [K, N]):
 * W4A16 and W8A16 the dequantized values in act_dtype, computed with exactly the
 * kernels' arithmetic (NVFP4: e2m1 x block scale; the tensor scale multiplies
 * the fp32 sum); MXFP4 the e4m3 byte of each e2m1 code (the e8m0 block
 * scale is applied inside the MMA).  Columns are in the standard order for
 * gated layers too (the pack's gate/up interleave is undone).
 * Source: the dequantization-and-scaling component (kinachrichten.com,
 * "Kompilierzeiten und geraetespezifisches Tuning"), exposed so that tests
 * can check it bit for bit.
 */
qgemm_status qgemm_debug_dequant(const qgemm_layer_config* layer, const void* packed,
                                 void* out_kn, void* stream);

/*
 * Synchronizes `stream`, reads the workspace status word written by the GEMM
 * kernels, clears it and returns QGEMM_OK, QGEMM_ERR_TIMEOUT (a bounded wait
 * gave up) or QGEMM_ERR_DEVICE.  After a timeout the caller must zero the
 * workspace again (qgemm_workspace_init) before reuse.
 * The pages have no counterpart: this reports the bounded waits of the
 * kernels.
 */
qgemm_status qgemm_check_status(void* workspace, void* stream);

/*
 * Wait limit, in nanoseconds, that kernels launched afterwards by this process
 * give each internal wait before they abandon the launch and report
 * QGEMM_ERR_TIMEOUT (default 1e9).  Exists to test the timeout path.
 */
void qgemm_set_wait_limit_ns(uint64_t ns);

/*
 * Checked build.  libqgemm_checked.so is this library compiled with
 * QGEMM_CHECKED: before every global-memory access whose index the kernels
 * compute from their inputs or schedule (weight blocks, split-K counters and
 * accumulators, cluster receive slots, output rows and columns, bias and
 * activation-scale entries, the MoE permutation, gather and combine indexes),
 * the kernel tests the index against the problem's extents.  A failed test
 * skips the access and records QGEMM_ERR_DEVICE instead of trapping: in the
 * workspace status word (read by qgemm_check_status or
 * qgemm_noalloc_check_status) for the GEMM kernels, and in a word of the
 * library (read by qgemm_checked_status) for the MoE support kernels.  Results
 * of inputs that pass every test are bitwise those of the unchecked build.
 *   qgemm_checked_build     1 in the checked build, 0 otherwise.
 *   qgemm_checked_status    synchronizes `stream`, reads and clears the word
 *                           of the MoE support kernels: QGEMM_OK or
 *                           QGEMM_ERR_DEVICE (QGEMM_OK always in the
 *                           unchecked build).
 *   qgemm_checked_selftest  launches on `stream` one index test that fails by
 *                           construction (nothing is accessed), recording into
 *                           the workspace status word (device, 16-byte
 *                           aligned); QGEMM_ERR_UNSUPPORTED in the unchecked
 *                           build.
 * The pages have no counterpart: this is a debugging aid of this library.
 */
int qgemm_checked_build(void);
qgemm_status qgemm_checked_status(void* stream);
qgemm_status qgemm_checked_selftest(void* workspace, void* stream);

/*
 * The compatibility record of a call: writes into buf (NUL-terminated, at most
 * len bytes) which kernel variant and tuning the heuristic picks for this
 * (layer, compute, m) on the current device, or why the combination is
 * rejected.  Returns the status the corresponding run call would return for
 * the configuration checks.
 * Source: the compatibility record that names the weight representation,
 * activation type, device and shapes and which implementation serves them
 * (retrivium.ai, "humming-format-kernel-contract-release", section "A
 * compatibility example").
 */
qgemm_status qgemm_describe_plan(const qgemm_layer_config* layer,
                                 const qgemm_compute_config* compute, int64_t m, char* buf,
                                 size_t len);

/* Static string naming a status code. */
const char* qgemm_status_string(qgemm_status status);

/* Reason for the last non-OK status returned on this thread ("" if none). */
const char* qgemm_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H_ */
