// Library-internal declarations shared by the C ABI layer and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#ifdef __CUDACC__
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#endif

namespace qg {

constexpr int kTileN = 128;       // output features per tile (MMA M extent)
constexpr int kTileK = 128;       // K per pipeline stage
constexpr int kTileBytes = kTileN * kTileK / 2;   // packed 4-bit weights per tile
constexpr int kNumThreads = 512;  // 16 warps: weights, MMA, TMEM, activations, 8 dequant, 4 epilogue
constexpr int kASlots = 4;        // TMEM slots for dequantized weight tiles
constexpr int kASlotCols = 64;    // TMEM columns per slot (128 K x 16 bit)
// k-tiles ("units") per activation slot for a token tile of bt rows: a slot
// is filled by one TMA box, so small token tiles group several k-tiles to
// keep every copy large.
__host__ __device__ constexpr int units_per_stage(int bt) { return bt <= 32 ? 4 : bt == 64 ? 2 : 1; }
// k-tiles per weight slot (one bulk copy of their packed blocks).
__host__ __device__ constexpr int weight_units_per_slot(int bt) { return bt <= 32 ? 4 : 2; }
constexpr int kEpiStageBytes = 4 * 2 * 16 * 32 * 2;   // output staging: 4 warps x 2 x 16 x 32
constexpr int kStatusTimeout = 1;
constexpr int kStatusDevice = 2;
// Checked build (compiled with -DQGEMM_CHECKED): the kernels test the
// global-memory indexes they compute from their inputs and their schedule
// against the problem's extents before each access.  A failed test skips the
// access and records kStatusDevice | kStatusCheck (in the workspace status
// word, or in the checked-build word of kernels that have no workspace)
// instead of trapping; the unchecked build compiles the tests away.
#ifdef QGEMM_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
constexpr int kStatusCheck = 1 << 24;
__device__ __forceinline__ bool qg_check(bool ok, int* word) {
  if constexpr (kChecked) {
    if (!ok) {
      atomicOr(word, kStatusDevice | kStatusCheck);
      return false;
    }
  }
  return true;
}
// The checked-build word of the kernels without a workspace (permute, gather,
// combine): read and cleared by qgemm_checked_status.
int checked_word_read_and_clear();
// Launches a kernel whose one index test fails on purpose (no access is made).
cudaError_t launch_check_selftest(int* word, cudaStream_t stream);
// With kStatusTimeout, the tcgen05 kernel also sets the bit of the wait that
// gave up first in its CTA (bits 8 and up), for the error message.
constexpr int kSiteWeightSlot = 1 << 8;     // weight producer: a free weight slot
constexpr int kSiteActSlot = 1 << 9;        // activation producer: a free activation slot
constexpr int kSiteScaleFactors = 1 << 10;  // MMA: the W4A8 B scale factors
constexpr int kSiteAccEmpty = 1 << 11;      // MMA: a free accumulator
constexpr int kSiteActFull = 1 << 12;       // MMA: activations landed
constexpr int kSiteDequantFull = 1 << 13;   // MMA: a dequantized weight tile
constexpr int kSiteWeightFull = 1 << 14;    // dequant: weights landed
constexpr int kSiteTmemSlot = 1 << 15;      // dequant: a free tensor-memory slot
constexpr int kSiteAccFull = 1 << 16;       // epilogue: a finished accumulator
constexpr int kSiteClusterRecv = 1 << 17;   // epilogue: the cluster peers' slices
constexpr int kSiteSplitCount = 1 << 18;    // split-K finisher: the contributors' count
constexpr int kSiteSplitCopy = 1 << 19;     // split-K finisher: the copied sum
constexpr int kSiteW4A4Slot = 1 << 20;      // W4A4 producer: a free pipeline stage
constexpr int kSiteW4A4Full = 1 << 21;      // W4A4 scale stager / MMA: a landed stage
constexpr int kSiteW4A4Scales = 1 << 22;    // W4A4 MMA: a stage's scale factors in TMEM
constexpr int kSiteW4A4Acc = 1 << 23;       // W4A4 epilogue: the finished accumulator
constexpr int kMaxExperts = 1024;      // grouped GEMM
constexpr int kMaxPermuteExperts = 256; // MoE permutation

// Workspace layout (bytes): [0, 256) status word and padding; then `counters`
// int32 per 32-column quarter of every output tile; then fp32 partial tiles, two per CTA.
struct WorkspaceLayout {
  size_t counters_off, counters_bytes, partials_off, partials_bytes;
  // W4A8 with bf16 activations above the small-M kernel: the e4m3 codes
  // [rows, K] and the per-row fp32 scales the library quantizes into (last,
  // outside the part that must start zeroed; aq_bytes 0 otherwise)
  size_t aq_off, aq_bytes, aq_scale_off;
  size_t total;
};

WorkspaceLayout workspace_layout(int64_t max_tiles, int grid, int block_tok);

// Division by a run-time invariant divisor d >= 1 with one multiply-high, an
// add and a shift (Granlund and Montgomery, "Division by invariant integers
// using multiplication", PLDI 1994): with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1, n / d = (umulhi(n, m) + n) >> s for
// every 0 <= n < 2^31 (the sum then stays below 2^32).
struct FastDiv {
  uint32_t d, mul, shift;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  uint32_t s = 0;
  while (s < 32 && (uint64_t(1) << s) < d) ++s;
  f.shift = s;
  f.mul = (uint32_t)(((uint64_t(1) << 32) * ((uint64_t(1) << s) - d)) / d + 1);
  return f;
}

struct W4A16Params {
  const uint8_t* w;          // packed blocks of all experts: [weights][scales][zeros]
  const uint16_t* bias;      // [E, N] or null
  uint16_t* c;               // [rows, N], or [rows, N/2] when gated
  const float* a_scale;      // W4A8: per-row activation scales [rows], else null
  int rows;                  // M (dense) or total permuted rows (grouped)
  int n, k;
  int kt, nt;                // k-tiles, n-tiles
  int st;                    // scale groups per k-tile
  int group;                 // group size
  int sg_shift;              // scale group of 32-wide k chunk j is j >> sg_shift
  int has_zp;
  int gated;                 // 1: SiLU-gated output from interleaved gate/up rows
  const float* t_scales;     // NVFP4: per-expert fp32 tensor scales (packed buffer tail)
  int split_cap;             // most CTAs sharing a tile's K range (0: no cap)
  const int* expert_offsets; // device [E+1] or null (dense)
  int num_experts;
  long long w_expert_stride; // bytes between experts' packed blocks
  int block_bytes;           // one (n-tile, k-tile) block: 8192 + scale + zero bytes
  int s_off, z_off;          // scales and zero points inside a block
  float* partials;           // fixed-order: two slots per CTA; atomic: one per split tile
  int deterministic;         // 1: fixed-order split-K reduction
  int* counters;
  int* status;
  long long max_tiles;
  int x_stages, x_bytes;     // activation ring: slots, bytes per slot (1 KB multiple)
  int w_stages, w_bytes, rw; // weight ring: slots, bytes per slot, k-tiles per slot
  int off_w, off_epi, off_bar;   // shared-memory offsets of the weight ring, staging, barriers
  int w_reuse;               // 1: several token tiles read each weight block (keep it in L2)
  int fix_smem;              // 1: the activation ring can hold a split tile's fp32 sum
  int last_stage;            // 1: ... and, after it, 2 KB per 16-row chunk of a tile
  // dense schedule, computed on the host: tiles, whole waves, stream-K units,
  // CTAs sharing them, and dividers for the schedule's invariant divisors
  int sk_t, sk_w, sk_u, sk_gs;
  FastDiv div_kt, div_nt, div_gs, div_u;
  int smem_bytes;            // total dynamic shared memory
  // cluster split (dense): S > 1 CTAs per tile in clusters of S, one K slice
  // each, reduced through distributed shared memory into receive slots at
  // off_recv; 0 otherwise
  int cluster, off_recv;
  unsigned long long wait_limit_ns;
};

// The small-M kernel (mma.sync, M <= 16, INT4 / UINT4): one cluster of
// `splits` CTAs per n-tile, each CTA a contiguous K slice of at most nk_max
// k-tiles streamed through a ring of `ring` weight slots; the slices' fp32
// partials are summed through distributed shared memory.  The workspace holds
// only the status word.
struct W4A16MmaParams {
  const uint8_t* w;          // packed blocks (one expert)
  const uint16_t* a;         // activations [m, k]
  uint16_t* c;               // output [m, n]
  const uint16_t* bias;      // [n] or null
  int* status;               // workspace status word (bounded waits report here)
  int m, n, k, kt, nt;
  int splits;                // K slices per n-tile = CTAs per cluster (1, 2, 4, 8, 16)
  int ring;                  // weight slots per CTA
  int nk_max;                // most k-tiles in one slice
  int block_bytes, s_off, z_off, sg_shift, has_zp;
  int mx;                    // 1: W4A8 (MXFP4 weights, e4m3 activations, bf16 output)
  const float* a_scale;      // W4A8: per-row activation scales [m] (quant_act: unused)
  int quant_act;             // W4A8: 1 = a is bf16 and the kernel quantizes it per row
  int f16s;                  // 1: bf16 activations with fp16 scales
  int nv;                    // 1: NVFP4 weights (16-bit block scales in the blocks)
  const float* t_scales;     // NVFP4: the fp32 tensor scale (the packed buffer's tail)
  unsigned long long wait_limit_ns;
};
// tmap_a: activations as {128 bytes of k, m rows, chunks}, 128-byte swizzle,
// box {128 bytes, 8 or 16 rows, nk_max k-tiles of chunks} (16-bit, also bf16
// activations that the kernel quantizes: 64 k per chunk, two chunks a k-tile;
// e4m3: 128 k, one)
cudaError_t launch_w4a16_mma(const CUtensorMap& tmap_a, const W4A16MmaParams& p, bool fp16,
                             cudaStream_t stream);
// dynamic shared memory of one small-M CTA (rows: 8 for M <= 8, else 16;
// elem_bytes: 2 for 16-bit activations, 1 for e4m3; quant: bf16 activations
// quantized to e4m3 in the kernel)
int mma_smem_bytes(int block_bytes, int ring, int nk_max, int rows, int elem_bytes,
                   bool quant = false);

// Clusters of S CTAs of the dense tcgen05 kernel (token tile bt, format fmt,
// smem bytes of dynamic shared memory) that can be resident at once; 0 if
// unknown.
int w4a16_max_clusters(int bt, int fmt, int S, int smem);

// W4A4 (NVFP4 weights x NVFP4 activations, kind::mxf4nvf4): one CTA per
// (token tile, 128-feature tile), the whole K range in 256-k stages.  The
// four tensor maps are uint8: weight codes {K/2, N} and activation codes
// {K/2, M} in 128-byte boxes with the 128-byte swizzle, weight and
// activation block scales {K/16, N} and {K/16, M} in 16-byte boxes.
struct W4A4Params {
  int m, n, k;               // k a multiple of 256
  int kt, nt, mt;            // 256-k stages, 128-feature tiles, token tiles
  const float* a_ts;         // activation tensor scale (one fp32, device)
  const float* w_ts;         // weight tensor scale (one fp32, device)
  const uint16_t* bias;      // [n] bf16 or null
  uint16_t* c;               // [m, n] bf16
  int* status;               // workspace status word
  unsigned long long wait_limit_ns;
  // K split: each tile's stages in `splits` contiguous slices, one work item
  // each; with splits > 1 every slice writes its fp32 partial tile to
  // part[(tile * splits + slice) * BT * 128 ...] and the last of a tile's
  // slices to count in (per 32-feature quadrant, cnt[tile * 4 + q], zero at
  // launch) sums the slices in slice order and stores the output
  int splits;
  float* part;
  int* cnt;
  long long part_rows;       // rows of 128 fp32 the partials region holds (checked build)
  int cnt_words;             // counters the region holds (checked build)
};
constexpr int kW4A4TileK = 256;
int w4a4_smem_bytes(int block_tok);
cudaError_t launch_w4a4(const CUtensorMap& tm_w, const CUtensorMap& tm_a, const CUtensorMap& tm_ws,
                        const CUtensorMap& tm_as, const W4A4Params& p, int block_tok,
                        cudaStream_t stream);
// Per-token NVFP4 quantization of bf16 activations x[m, k] (k % 16 == 0):
// codes [m, k/2] (k = 2i in the low nibble of byte i), e4m3 block scales
// [m, k/16]; a_ts is the caller's fp32 tensor scale on the device.  The
// kernel also sets zero_words[0 .. n_zero) to zero (the W4A4 GEMM's K-split
// counters; null and 0 for none).
cudaError_t launch_act_quant_nvfp4(const uint16_t* x, int64_t m, int64_t k, const float* a_ts,
                                   uint8_t* codes, uint8_t* sb, cudaStream_t stream,
                                   int* zero_words = nullptr, int n_zero = 0);

// Host-side plan for one W4A16 launch.
int device_sm_count();
// fmt: 0 = W4A16 bf16, 1 = W4A16 fp16, 2 = W4A8 (MXFP4 x e4m3, bf16 out),
//      3 = NVFP4 weights x bf16, 4 = NVFP4 weights x fp16,
//      5 = W4A16 bf16 with fp16 scales, 6 / 7 = W8A16 bf16 / fp16
cudaError_t launch_w4a16(const CUtensorMap& tmap_a, const CUtensorMap& tmap_c,
                         const W4A16Params& p, int block_tok, int fmt, bool grouped, int grid,
                         cudaStream_t stream);

cudaError_t launch_repack_mxfp4(const uint8_t* codes, const uint8_t* scales, uint8_t* packed,
                                int64_t n, int64_t k, int experts, int gated, cudaStream_t stream);

cudaError_t launch_debug_mx_codes(const uint8_t* w, uint8_t* out_kn, int64_t n, int64_t k,
                                  int gated, cudaStream_t stream);

// Packed block of one (n-tile, k-tile): the codes (8192 bytes of 4-bit
// codes, 16384 bytes of 8-bit ones), then the scales (128 * st 16-bit words;
// MXFP4: 128 32-bit words), then the zero points (128 * st bytes) when the
// format has them.
__host__ __device__ constexpr int packed_code_bytes(bool w8) {
  return w8 ? 2 * kTileBytes : kTileBytes;
}
__host__ __device__ constexpr int packed_scale_bytes(bool mx, int st) {
  return mx ? kTileN * 4 : st * kTileN * 2;
}
__host__ __device__ constexpr int packed_block_bytes(bool mx, int st, bool zp, bool w8 = false) {
  return packed_code_bytes(w8) + packed_scale_bytes(mx, st) + (zp ? st * kTileN : 0);
}

// Gated layers: packed row r of n-tile nt holds standard column
// (r & 1) * N/2 + 64 nt + r/2, so gate column i and up column N/2 + i sit on
// neighbouring rows (neighbouring lanes of the epilogue) of one tile.
__host__ __device__ inline int glu_source_col(int nt, int r, int n) {
  return (r & 1) * (n >> 1) + nt * (kTileN / 2) + (r >> 1);
}
__host__ __device__ inline int packed_source_col(int nt, int r, int n, int gated) {
  return gated ? glu_source_col(nt, r, n) : nt * kTileN + r;
}

#ifdef __CUDACC__
// SiLU gate of one (gate, up) pair in fp32: g / (1 + e^-g) * u with the
// hardware exponential and the approximate divide (relative error ~1e-6,
// far below the bf16 rounding that follows; e^-g = inf gives the limit 0).
// The GEMM epilogue runs it beside the dequant warps, where an IEEE exp and
// divide would cost several times the issue slots.  Each operation is
// rounded on its own (no contraction), so the fused GEMM epilogue and the
// standalone kernel produce the same bits from the same rounded inputs.
__device__ __forceinline__ float silu_mul_f32(float g, float u) {
  return __fmul_rn(__fdividef(g, __fadd_rn(1.f, __expf(-g))), u);
}

// bf16 activations with fp16 scales: w^ = bf16((q - z) * s), one rounding.
// The scale is split into s_hi, its leading 8 significant bits (a bf16), and
// the rest s_lo = s - s_hi, which has at most 3 significant bits (an fp16 has
// 11) and the sign of s, so it is a bf16 too.  With d = q - z (an integer of
// at most 4 bits, exact in bf16), t = d * s_lo has at most 7 significant bits
// and is exact, and fma(d, s_hi, t) rounds the exact d * s once.  Zero
// results carry the sign of d * s: both terms are then zeros of that sign.
// Four e2m1 codes (bits 0-15, code c at bits 4c..4c+3) -> two packed 16-bit
// pairs of their values, exactly (every e2m1 value is an fp16 and a bf16
// value): p0 = (code 0, code 1), p1 = (code 2, code 3), the lower k in the low
// half.  prmt looks up the bytes of each code magnitude's 16-bit pattern in
// 8-entry byte tables (fp16: the low byte is always 0), a sign-replicating
// prmt turns each code's sign bit into bit 6 of a byte, and one lop3 moves it
// into the sign of the high byte.
template <bool FP16>
__device__ __forceinline__ void e2m1x4_pairs(uint32_t c16, uint32_t& p0, uint32_t& p1) {
  const uint32_t sel = c16 & 0x7777u;
  uint32_t sgn, hi;
  asm("prmt.b32 %0, %1, %1, %2;" : "=r"(sgn) : "r"(0x80808080u), "r"(c16));
  if constexpr (FP16) {   // high bytes of fp16 0, 0.5, 1, 1.5 | 2, 3, 4, 6
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(0x3E3C3800u), "r"(0x46444240u), "r"(sel));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(hi) : "r"(sgn << 1), "r"(0x80808080u), "r"(hi));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p0) : "r"(hi), "r"(0u), "r"(0x1404u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p1) : "r"(hi), "r"(0u), "r"(0x3424u));
  } else {                // bf16: high and low bytes of the same eight values
    uint32_t lo;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(0x3F3F3F00u), "r"(0x40404040u), "r"(sel));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(0xC0800000u), "r"(0xC0804000u), "r"(sel));
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(hi) : "r"(sgn << 1), "r"(0x80808080u), "r"(hi));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p0) : "r"(lo), "r"(hi), "r"(0x5140u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p1) : "r"(lo), "r"(hi), "r"(0x7362u));
  }
}

__device__ __forceinline__ void split_f16_scale(uint16_t bits, uint32_t& hi2, uint32_t& lo2) {
  const float s = __half2float(__ushort_as_half(bits));
  uint32_t hi, lo;
  if (isfinite(s)) {
    const uint32_t sb = __float_as_uint(s);
    const float rest = s - __uint_as_float(sb & 0xFFFF0000u);   // exact
    hi = sb >> 16;
    lo = (__float_as_uint(rest) >> 16) | ((sb >> 16) & 0x8000u);
  } else {   // inf or NaN: the products d * s of IEEE arithmetic
    const __nv_bfloat16 b = __float2bfloat16_rn(s);
    hi = *reinterpret_cast<const uint16_t*>(&b);
    lo = 0;
  }
  hi2 = hi * 0x00010001u;
  lo2 = lo * 0x00010001u;
}
#endif

// code_bits 4: INT4 / UINT4 (qweight int32 [K/8, N], qzeros [K/g, N/8]);
// 3: INT3 / UINT3 bit streams (qweight int32 [3K/32, N], qzeros [K/g, 3N/32]),
// repacked into the same 4-bit blocks.
cudaError_t launch_repack_w4(const int32_t* qweight, const uint16_t* scales,
                             const int32_t* qzeros, uint8_t* packed, int64_t n, int64_t k,
                             int group, int signed_q, int experts, int gated, int code_bits,
                             cudaStream_t stream);
// INT8 / UINT8: standard qweight int32 [K/4, N], scales [K/g, N], qzeros
// int32 [K/g, N/4] or null -> packed blocks of 16384 code bytes.
cudaError_t launch_repack_w8(const int32_t* qweight, const uint16_t* scales,
                             const int32_t* qzeros, uint8_t* packed, int64_t n, int64_t k,
                             int group, int signed_q, int experts, int gated,
                             cudaStream_t stream);

cudaError_t launch_debug_dequant(const uint8_t* packed, uint16_t* out, int64_t n, int64_t k,
                                 int group, int has_zp, bool fp16, bool nv, bool f16s,
                                 bool w8, int gated, cudaStream_t stream);

cudaError_t launch_repack_nvfp4(const uint8_t* codes, const uint8_t* scales,
                               const float* tensor_scales, uint8_t* packed, int64_t n, int64_t k,
                               int experts, bool fp16, int gated, cudaStream_t stream);

cudaError_t launch_act_quant_fp8(const uint16_t* x, int64_t m, int64_t k, uint8_t* a8,
                                 float* scale, cudaStream_t stream);

cudaError_t launch_moe_permute(const int32_t* ids, int64_t t, int topk, int e, int32_t* offsets,
                               int32_t* perm, int32_t* inv_perm, const uint16_t* a,
                               uint16_t* a_perm, int64_t hidden, cudaStream_t stream);

cudaError_t launch_silu_mul(const uint16_t* gu, int64_t rows, int64_t inter, uint16_t* h,
                            cudaStream_t stream);

cudaError_t launch_combine(const uint16_t* y2, const int32_t* inv_perm, const float* w, int64_t t,
                           int topk, int64_t hidden, uint16_t* y, cudaStream_t stream);

// Host helpers shared with the allocation-free entry point: set the calling
// thread's error message, and the bytes of a dense GEMM's workspace that must
// be zero before a launch (status word and split-K counters) and in total.
int set_last_error(int status, const char* message);
int dense_workspace_bytes(const void* layer, const void* compute, const void* tuning, int64_t m,
                          size_t* must_clear, size_t* total);
// qgemm_run that, once every argument check has passed and just before the
// launch, zeroes the first clear_bytes of the workspace on the stream (0: no
// clear).  A call rejected by a check queues nothing.
int run_dense_clearing(const void* layer, const void* compute, const void* tuning, int64_t m,
                       const void* a, const float* a_scale, const void* packed, const void* bias,
                       void* c, void* workspace, size_t ws_bytes, size_t clear_bytes,
                       cudaStream_t stream);

bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    const uint64_t dims[3], const uint64_t strides_bytes[2],
                    const uint32_t box[3], CUtensorMapSwizzle swizzle);

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                    uint32_t box_outer, CUtensorMapSwizzle swizzle);

}  // namespace qg
