// W4A16 GEMM for sm_103a: C[M, N] = A[M, K] . W^[K, N], W^ = adt((q - z) * s).
//
// The Humming pages assemble their kernels from scheduling, data movement,
// dequantization/scaling, tensor-core compute and output processing
// (kinachrichten.com, "Kompilierzeiten und geraetespezifisches Tuning"), with
// a TMA + UMMA pipeline for larger batches and a multi-stage cp.async + MMA
// pipeline for small ones (same article, section "Wie die Architektur
// funktioniert").  This kernel is the B300 design of those five components
// for every M and format (the cp.async + mma.sync kernel in w4a16_mma.cu
// takes dense INT4/UINT4 GEMMs of at most 16 rows):
//
//   swap-AB:  the MMA computes D[n, m] = W^[n, :] . A[m, :], so the 128 output
//             features of a tile are the MMA M extent and the tokens are the
//             MMA N extent (16 .. 128), which keeps the tensor core busy at
//             tiny M.
//   data movement (warp 0): plain bulk copies of the pre-tiled 4-bit weight,
//             scale and zero blocks, and a TMA tensor load (128-byte swizzle)
//             of the activation tile, into a ring of shared-memory stages.
//   dequant (warps 4..11): each thread owns one output feature (one TMEM
//             lane), unpacks 32 nibbles per 16-byte vector with LOP3 against a
//             magic exponent, subtracts (magic + z) exactly and multiplies by
//             the scale once (the single rounding of the dequant definition),
//             and stores the 16-bit pairs straight into tensor memory, where
//             tcgen05.mma reads them as its A operand.  No shared-memory
//             round trip for the dequantized weights.
//   tensor core (warp 1): one thread issues tcgen05.mma kind::f16 with A in
//             TMEM and the activation tile as the shared-memory B operand,
//             accumulating in fp32 in TMEM (two accumulator buffers).
//   output (warps 12..15): tcgen05.ld of the accumulator, bias, rounding,
//             stores.  A tile whose K range was split is finished by the CTA
//             holding its first k-tiles (its last work item): the others add
//             their fp32 partials into an accumulator in L2 and count in; the
//             finisher adds the copied-in sum to its own partial in tensor
//             memory.  A fixed-order variant sums per-CTA partial slots.
//   scheduling: a persistent grid of at most one CTA per SM walks whole tiles
//             round-robin, then splits the remaining tiles' K ranges evenly
//             across all CTAs (stream-K), so every SM streams the same number
//             of weight bytes at any M.  The grouped (MoE) variant derives its
//             tiles from the expert offsets on the device.
//
// Every wait is bounded (see mbar_wait); a CTA that gives up records a
// timeout in the workspace status word and drains its own copies before it
// frees tensor memory and exits.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <map>
#include <mutex>
#include <tuple>

#include "internal.h"
#include "ptx.cuh"

namespace qg {

namespace {

struct WorkItem {
  int tile;
  int k0, k1;
};

__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
  return (int)((__umulhi((unsigned)n, f.mul) + (unsigned)n) >> f.shift);
}

// Whole tiles round-robin (waves), then an even split of the remaining tiles'
// K-tiles ("units") across the first Gs = min(G, U) CTAs, so that every CTA
// taking part in the split owns at least one unit; the CTAs that share a tile
// are then exactly cta_of_unit(first unit) .. cta_of_unit(last unit).  All
// arithmetic is 32-bit (the host bounds U * G below 2^31), and a dense GEMM's
// schedule constants and divisors come from the host: integer division is a
// long instruction sequence on the critical path of a kernel's start.
struct Schedule {
  int T;           // tiles
  int KT;          // k-tiles per tile
  int G, c;        // grid size, this CTA
  int W;           // full waves of whole tiles
  int U;           // stream-K units
  int Gs;          // CTAs sharing the stream-K units
  int it, u, u_end;
  bool fast;       // host-made dividers for Gs and U
  FastDiv dkt, dgs, du;

  // dense: everything from the host
  __device__ void init_dense(const W4A16Params& p, int c_) {
    T = p.sk_t;
    KT = p.kt;
    G = gridDim.x;
    c = c_;
    W = p.sk_w;
    U = p.sk_u;
    Gs = p.sk_gs;
    fast = true;
    dkt = p.div_kt;
    dgs = p.div_gs;
    du = p.div_u;
    start();
  }
  // grouped: the tile count is known only on the device
  __device__ void init(long long T_, const W4A16Params& p, int c_) {
    T = (int)T_;
    KT = p.kt;
    G = gridDim.x;
    c = c_;
    W = T / G;
    if (p.split_cap == 0 && W > 0 && T % G) --W;   // stream-K over the last two waves
    U = (T - W * G) * KT;
    Gs = U < G ? U : G;
    if (p.split_cap > 0 && U > 0) {   // each remaining tile to min(cap, G / r) CTAs
      const int r = U / KT;
      const int per = min(p.split_cap, G / r);
      Gs = min(Gs, r * per);
    }
    fast = false;
    dkt = p.div_kt;
    start();
  }
  __device__ void start() {
    it = 0;
    if (c < Gs) {
      u = sk_begin(c);
      u_end = sk_begin(c + 1);
    } else {
      u = u_end = 0;
    }
  }
  __device__ int sk_begin(int cta) const {
    return fast ? fdiv(cta * U, dgs) : (int)((unsigned)(cta * U) / (unsigned)Gs);
  }
  // CTA whose unit range holds unit uu.
  __device__ int cta_of_unit(int uu) const {
    const int x = (uu + 1) * Gs - 1;
    return fast ? fdiv(x, du) : (int)((unsigned)x / (unsigned)U);
  }

  __device__ bool next(WorkItem& wi) {
    if (it < W) {
      wi.tile = c + it * G;
      wi.k0 = 0;
      wi.k1 = KT;
      ++it;
      return true;
    }
    if (u >= u_end) return false;
    const int tl = fdiv(u, dkt);
    const int k0 = u - tl * KT;
    const int seg_end = min((tl + 1) * KT, u_end);
    wi.tile = W * G + tl;
    wi.k0 = k0;
    wi.k1 = k0 + (seg_end - u);
    u = seg_end;
    return true;
  }
};

struct SharedState {
  uint32_t tmem_base;
  int abort_flag;
  int pad0;
  int pad1;
  long long tiles;     // total tiles (grouped: from offsets)
};

template <int BT>
struct TileCoord {
  int e, row0, rows, nt;
};

}  // namespace

template <bool FP16>
__device__ __forceinline__ uint32_t dq_pair(uint32_t bits, uint32_t zero2, uint32_t scale2) {
  if constexpr (FP16) {
    __half2 x = *reinterpret_cast<__half2*>(&bits);
    __half2 zz = *reinterpret_cast<__half2*>(&zero2);
    __half2 ss = *reinterpret_cast<__half2*>(&scale2);
    __half2 r = __hmul2(__hsub2(x, zz), ss);
    return *reinterpret_cast<uint32_t*>(&r);
  } else {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&bits);
    __nv_bfloat162 zz = *reinterpret_cast<__nv_bfloat162*>(&zero2);
    __nv_bfloat162 ss = *reinterpret_cast<__nv_bfloat162*>(&scale2);
    __nv_bfloat162 r = __hmul2(__hsub2(x, zz), ss);
    return *reinterpret_cast<uint32_t*>(&r);
  }
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void red_release_add_gpu(int* addr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int* addr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

// Orders this thread's generic-proxy view of global memory before its later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* addr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(addr), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));   // (a & b) | c
  return d;
}

// 32 nibbles (one 16-byte vector of the tiled layout) -> 16 packed 16-bit pairs.
// Nibble positions p and p+4 of a word hold consecutive k, so one mask
// extracts a (k, k+1) pair straight into the low mantissa bits of two
// 16-bit floats whose exponent encodes `magic` (128 for bf16, 1024 for fp16,
// where the unit in the last place is 1): the pair reads magic + u exactly.
template <bool FP16>
__device__ __forceinline__ void dequant_vec(const uint4 v, uint32_t zero2, uint32_t scale2,
                                            uint32_t (&out)[16]) {
  constexpr uint32_t magic = FP16 ? 0x64006400u : 0x43004300u;
  const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t x = lop3_and_or(wds[w] >> (4 * i), 0x000F000Fu, magic);
      out[w * 4 + i] = dq_pair<FP16>(x, zero2, scale2);
    }
  }
}

// bf16 activations with fp16 scales (split_f16_scale, internal.h): one rounding.
__device__ __forceinline__ void dequant_vec_f16s(const uint4 v, uint32_t zero2, uint32_t hi2,
                                                 uint32_t lo2, uint32_t (&out)[16]) {
  constexpr uint32_t magic = 0x43004300u;
  const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
  const __nv_bfloat162 zz = *reinterpret_cast<const __nv_bfloat162*>(&zero2);
  const __nv_bfloat162 sh = *reinterpret_cast<const __nv_bfloat162*>(&hi2);
  const __nv_bfloat162 sl = *reinterpret_cast<const __nv_bfloat162*>(&lo2);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t x = lop3_and_or(wds[w] >> (4 * i), 0x000F000Fu, magic);
      const __nv_bfloat162 d = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&x), zz);
      __nv_bfloat162 r = __hfma2(d, sh, __hmul2(d, sl));
      out[w * 4 + i] = *reinterpret_cast<uint32_t*>(&r);
    }
  }
}

// 16 8-bit codes (one 16-byte vector of the tiled layout, k in byte order)
// -> 8 packed 16-bit pairs (k, k+1) of (u - z) * s, rounded once.  fp16: a
// prmt pairs two code bytes with 0x64 high bytes, so each half reads
// 1024 + u exactly (the unit in the last place is 1 up to 2048); the
// subtraction of 1024 + z is exact and the multiply rounds once.  bf16 has
// too few mantissa bits for 8-bit codes, so each code goes through fp32: a
// prmt places it in byte 1 of 0x47000000, which reads 2^15 + u; minus
// 2^15 + z is exact, the product with the scale (9 x 8 significant bits) is
// exact, and cvt.rn rounds each pair once.  Zero results carry the sign of
// the scale, as the products do.
template <bool FP16>
__device__ __forceinline__ void dequant_vec8(const uint4 v, uint32_t zero, uint32_t scale,
                                             uint32_t (&out)[8]) {
  const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    if constexpr (FP16) {
      uint32_t x0, x1;
      asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(x0) : "r"(wds[w]), "r"(0x64646464u));
      asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(x1) : "r"(wds[w]), "r"(0x64646464u));
      out[2 * w] = dq_pair<true>(x0, zero, scale);
      out[2 * w + 1] = dq_pair<true>(x1, zero, scale);
    } else {
      const float zf = __uint_as_float(zero), sf = __uint_as_float(scale);
      uint32_t x[4];
      asm("prmt.b32 %0, %1, %2, 0x7604;" : "=r"(x[0]) : "r"(wds[w]), "r"(0x47000000u));
      asm("prmt.b32 %0, %1, %2, 0x7614;" : "=r"(x[1]) : "r"(wds[w]), "r"(0x47000000u));
      asm("prmt.b32 %0, %1, %2, 0x7624;" : "=r"(x[2]) : "r"(wds[w]), "r"(0x47000000u));
      asm("prmt.b32 %0, %1, %2, 0x7634;" : "=r"(x[3]) : "r"(wds[w]), "r"(0x47000000u));
      float f[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) f[c] = __fmul_rn(__fsub_rn(__uint_as_float(x[c]), zf), sf);
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out[2 * w]) : "f"(f[1]), "f"(f[0]));
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out[2 * w + 1]) : "f"(f[3]), "f"(f[2]));
    }
  }
}

// 32 e2m1 codes (one 16-byte vector, k in nibble order, low nibble first) ->
// 32 e4m3 bytes, exactly (every e2m1 value is an e4m3 value).  prmt looks up
// the e4m3 byte of the 3-bit magnitude in an 8-entry byte table; a second
// prmt against 0x80 bytes turns each nibble's sign bit into bit 6 of its byte
// (sign-replicate mode), which the final lop3 moves into bit 7.
__device__ __forceinline__ uint32_t e2m1x4_to_e4m3x4(uint32_t c16) {
  constexpr uint32_t kLo = 0x3C383000u;   // e4m3 of 0, 0.5, 1, 1.5
  constexpr uint32_t kHi = 0x4C484440u;   // e4m3 of 2, 3, 4, 6
  uint32_t mag, sgn, out;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(mag) : "r"(kLo), "r"(kHi), "r"(c16 & 0x7777u));
  asm("prmt.b32 %0, %1, %1, %2;" : "=r"(sgn) : "r"(0x80808080u), "r"(c16));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(out) : "r"(sgn << 1), "r"(0x80808080u), "r"(mag));
  return out;   // ((sgn << 1) & 0x80808080) | mag
}

__device__ __forceinline__ void dequant_vec_mx(const uint4 v, uint32_t (&out)[8]) {
  const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    out[2 * w] = e2m1x4_to_e4m3x4(wds[w]);
    out[2 * w + 1] = e2m1x4_to_e4m3x4(wds[w] >> 16);
  }
}

template <bool FP16>
__device__ __forceinline__ uint32_t mul_pair(uint32_t bits, uint32_t scale2) {
  if constexpr (FP16) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&bits), *reinterpret_cast<__half2*>(&scale2));
    return *reinterpret_cast<uint32_t*>(&r);
  } else {
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&bits),
                               *reinterpret_cast<__nv_bfloat162*>(&scale2));
    return *reinterpret_cast<uint32_t*>(&r);
  }
}

// NVFP4: 32 e2m1 codes (one 16-byte vector, k in nibble order, low nibble
// first) -> 16 packed 16-bit pairs (k, k+1) of e2m1 value x block scale,
// exactly: every e2m1 x e4m3 product is a bf16 and an fp16 value (the code
// values by e2m1x4_pairs, internal.h).  Words 0-1 hold k 0..15 (scale sA2),
// words 2-3 k 16..31 (sB2).
template <bool FP16>
__device__ __forceinline__ void dequant_vec_nv(const uint4 v, uint32_t sA2, uint32_t sB2,
                                               uint32_t (&out)[16]) {
  const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {   // codes 4 hh .. 4 hh + 3 of the word
      uint32_t p0, p1;
      e2m1x4_pairs<FP16>(wds[w] >> (16 * hh), p0, p1);
      const uint32_t s2 = w < 2 ? sA2 : sB2;
      out[w * 4 + hh * 2] = mul_pair<FP16>(p0, s2);
      out[w * 4 + hh * 2 + 1] = mul_pair<FP16>(p1, s2);
    }
  }
}

template <bool FP16>
__device__ __forceinline__ uint16_t to_out(float v) {
  if constexpr (FP16) {
    __half h = __float2half_rn(v);
    return *reinterpret_cast<uint16_t*>(&h);
  } else {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&h);
  }
}

template <bool FP16>
__device__ __forceinline__ float from_out(uint16_t b) {
  if constexpr (FP16) {
    return __half2float(*reinterpret_cast<__half*>(&b));
  } else {
    return __bfloat162float(*reinterpret_cast<__nv_bfloat16*>(&b));
  }
}

// FMT: 0 = W4A16 bf16, 1 = W4A16 fp16, 2 = W4A8 (MXFP4 weights, e4m3
// activations with per-row fp32 scales, block-scaled MMA, bf16 output),
// 3 / 4 = NVFP4 weights with bf16 / fp16 activations, 5 = W4A16 bf16
// activations with fp16 scales, 6 / 7 = W8A16 (8-bit integer codes) with
// bf16 / fp16 activations.
//
// Shared memory holds two rings that turn over independently:
//   activation slots: RX = units_per_stage(BT) consecutive k-tiles ("units")
//     of one work item, one three-dimensional TMA box each; a slot goes back
//     to its producer when the MMAs that read it have completed;
//   weight slots: up to p.rw units' packed blocks (codes, scales, zero
//     points), one bulk copy each; a slot goes back as soon as the dequant
//     warps have read it into registers,
// so the weight stream runs ahead of the activations and of the tensor core,
// limited only by the weight ring's depth.
template <int BT, int FMT, bool GROUPED>
__global__ void __launch_bounds__(kNumThreads, 1)
    w4a16_kernel(const __grid_constant__ CUtensorMap tmap_a,
                 const __grid_constant__ CUtensorMap tmap_c, const W4A16Params p) {
  constexpr bool FP16 = FMT == 1 || FMT == 4 || FMT == 7;   // 16-bit activations and output: fp16
  constexpr bool MX = FMT == 2;                  // W4A8-MXFP4
  constexpr bool NV = FMT == 3 || FMT == 4;      // NVFP4 weights, 16-bit activations
  constexpr bool F16S = FMT == 5;                // bf16 activations, fp16 scales
  constexpr bool W8 = FMT == 6 || FMT == 7;      // 8-bit integer codes
  constexpr int RX = units_per_stage(BT);
  // tensor-memory columns: dequantized weight slots, then (MX) the A and B
  // scale factors, accumulators from column 256
  constexpr int kSlotCols = MX ? 32 : kASlotCols;
  constexpr uint32_t kSfaCol = 128, kSfbCol = 160, kAccCol = 256;
  constexpr uint32_t kActUnit = BT * kTileK * (MX ? 1 : 2);   // bytes of one unit's activations
  // accumulator buffers of BT columns from column 256: two (the epilogue of
  // one tile overlaps the next tile's MMAs) up to 128 tokens, one at 256
  constexpr int NACC = BT == 256 ? 1 : 2;
  static_assert(BT <= 128 || !MX, "256-token tiles take 16-bit formats only");

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled operand tiles
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int SX = p.x_stages, SW = p.w_stages, RW = p.rw;
  uint8_t* x_base = smem;                    // SX slots of p.x_bytes (1 KB multiples)
  uint8_t* w_base = smem + p.off_w;          // SW slots of p.w_bytes
  uint16_t* epi_stage = reinterpret_cast<uint16_t*>(smem + p.off_epi);   // 4 warps x 2 x 16 x 32
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* x_full = bars;
  uint64_t* x_empty = x_full + SX;
  uint64_t* w_full = x_empty + SX;
  uint64_t* w_empty = w_full + SW;
  uint64_t* a_full = w_empty + SW;
  uint64_t* a_empty = a_full + kASlots;
  uint64_t* acc_full = a_empty + kASlots;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* sfb_ready = drain + 1;
  uint64_t* fix_bar = sfb_ready + 1;   // one per epilogue warp: split-K sum copied in
  uint64_t* recv_full = fix_bar + 4;   // cluster split: the peers' slices have landed
  SharedState* sh = reinterpret_cast<SharedState*>(recv_full + 1);
  int* mt_prefix = reinterpret_cast<int*>(sh + 1);     // grouped: m-tile prefix [E+1]
  int* offs = mt_prefix + (GROUPED ? (p.num_experts + 1) : 0);   // grouped: offsets [E+1]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sh->abort_flag;
  const uint64_t lim = p.wait_limit_ns;
  const int blk_bytes = p.block_bytes;   // packed block: codes, scales, zero points

  auto coords = [&](int tile) {
    TileCoord<BT> tc;
    const int mtg = fdiv(tile, p.div_nt);
    tc.nt = tile - mtg * p.nt;
    if constexpr (GROUPED) {
      int lo = 0, hi = p.num_experts;   // find e: mt_prefix[e] <= mtg < mt_prefix[e+1]
      while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (mt_prefix[mid] <= mtg) lo = mid; else hi = mid;
      }
      tc.e = lo;
      tc.row0 = offs[lo] + (mtg - mt_prefix[lo]) * BT;
      tc.rows = min(BT, offs[lo + 1] - tc.row0);
    } else {
      tc.e = 0;
      tc.row0 = mtg * BT;
      tc.rows = min(BT, p.rows - tc.row0);
    }
    return tc;
  };
  // waits for every copy a producer issued into its ring to land, so that no
  // copy is still writing shared memory when the CTA exits
  auto drain_ring = [&](uint64_t* full, int S, int issued) {
    for (int st = 0; st < S && st < issued; ++st) {
      const int last = st + ((issued - 1 - st) / S) * S;
      volatile int no_abort = 0;
      mbar_wait(&full[st], (uint32_t)((last / S) & 1), &no_abort, nullptr, 100000000ull, 0);
    }
  };

  // Dense GEMMs: the first weight slot goes out before anything else, from
  // the host-made schedule, so that the weight stream starts within a few
  // hundred instructions of the launch.
  bool first_issued = false;
  if (!GROUPED && threadIdx.x == 0) {
    mbar_init(&w_full[0], 1);
    mbar_init(&w_empty[0], 8);
    fence_barrier_init();
    Schedule s0;
    s0.init_dense(p, blockIdx.x);
    WorkItem w0;
    if (s0.next(w0)) {
      const int nt0 = w0.tile - fdiv(w0.tile, p.div_nt) * p.nt;
      const int r = min(RW, w0.k1 - w0.k0);
    if (qg_check(nt0 >= 0 && nt0 < p.nt && w0.k0 >= 0 && w0.k0 + r <= p.kt, p.status)) {
      mbar_arrive_expect_tx(&w_full[0], r * blk_bytes);
      bulk_load(w_base, p.w + ((long long)nt0 * p.kt + w0.k0) * blk_bytes, r * blk_bytes,
                &w_full[0], p.w_reuse ? policy_evict_normal() : policy_evict_first());
      first_issued = true;
    }
    }
  }
  if (warp == 0) {
    // barrier initialization spread over the warp's lanes: lane i sets up
    // barrier i of the contiguous array (arrival counts by the array it is in);
    // a dense GEMM's first weight slot barriers are set up already
    const int nb = 2 * SX + 2 * SW + 2 * kASlots + 4 + 2 + 4 + 1;
    for (int i = lane; i < nb; i += 32) {
      if (!GROUPED && (i == 2 * SX || i == 2 * SX + SW)) continue;
      uint32_t count = 1;
      int j = i - 2 * SX;
      if (j >= SW && j < 2 * SW) count = 8;                 // w_empty: every dequant warp
      j -= 2 * SW;
      if (j >= 0 && j < kASlots) count = 4;                 // a_full: one per lane quadrant
      j -= 2 * kASlots;
      if (j == 2 || j == 3) count = 4;                      // acc_empty
      if (j == 5) count = 4;                                // sfb_ready
      mbar_init(&bars[i], count);
    }
    if (lane == 0) sh->abort_flag = 0;
    fence_barrier_init();
    if (!GROUPED && p.cluster > 1) {
      // cluster split: this CTA finishes the 16-row chunks u = 32 q / 16 +
      // chunk with u % S == its rank and receives the S - 1 other slices of
      // each (2 KB apiece; chunks past the tile's rows are not sent)
      __syncwarp();
      if (lane == 0) {
        const int S = p.cluster, sl = (int)(blockIdx.x % (unsigned)S);
        const int tile = (int)(blockIdx.x / (unsigned)S);
        const int rows = min(BT, p.rows - fdiv(tile, p.div_nt) * BT);
        const int nlive = (rows + 15) / 16;
        int owned = 0;
        for (int u = 0; u < 4 * (BT / 16); ++u)
          if (u % S == sl && u % (BT / 16) < nlive) ++owned;
        mbar_arrive_expect_tx(recv_full, (uint32_t)(owned * (S - 1) * 2048));
      }
    }
  }
  if (warp == 2) {
    tmem_alloc(&sh->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 3) {
    if constexpr (GROUPED) {
      // m-tile prefix over experts, from the device-side offsets (written by
      // the previous grid on the stream, so wait for it first).  Offsets are
      // caller data: clamped to [0, rows] and made monotone (a running max)
      // so that no tile reaches outside the row range; both passes are warp
      // scans, 32 experts at a time.
      grid_dependency_wait();
      const int E = p.num_experts;
      int carry = 0;
      for (int x0 = 0; x0 <= E; x0 += 32) {
        const int x = x0 + lane;
        int v = x <= E ? min(max(p.expert_offsets[x], 0), p.rows) : p.rows;
        if (x == 0) v = 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, v, d);
          if (lane >= d) v = max(v, t);
        }
        v = max(v, carry);
        if (x <= E) offs[x] = v;
        carry = __shfl_sync(0xffffffffu, v, 31);
      }
      __syncwarp();
      int acc = 0;
      for (int x0 = 0; x0 < E; x0 += 32) {
        const int x = x0 + lane;
        const int c = x < E ? (offs[x + 1] - offs[x] + BT - 1) / BT : 0;
        int incl = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += t;
        }
        if (x < E) mt_prefix[x + 1] = acc + incl;
        acc += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        mt_prefix[0] = 0;
        long long T = (long long)acc * p.nt;
        if (T > p.max_tiles) {   // offsets inconsistent with the workspace bound
          atomicOr(p.status, kStatusDevice);
          T = 0;
        }
        sh->tiles = T;
      }
    } else {
      if (lane == 0) sh->tiles = (long long)((p.rows + BT - 1) / BT) * p.nt;
    }
  }
  // Start-up barrier.  For a dense GEMM the weight producer only arrives (it
  // needs neither tensor memory nor the grouped tile table), so the weight
  // stream starts while the other warps wait for the allocation.
  tc_fence_before();
  if (!GROUPED && warp == 0) {
    __syncwarp();
    asm volatile("bar.arrive 1, %0;" ::"n"(kNumThreads) : "memory");
  } else {
    asm volatile("bar.sync 1, %0;" ::"n"(kNumThreads) : "memory");
  }
  tc_fence_after();
  // cluster split: every receive barrier of the cluster is set up once this
  // barrier phase completes (waited for before the first send)
  bool cl_waited = false;
  if (!GROUPED && p.cluster > 1) cluster_arrive();
  const uint32_t tmem_base = (!GROUPED && warp == 0) ? 0u : sh->tmem_base;
  const long long T = (!GROUPED && warp == 0)
                          ? (long long)((p.rows + BT - 1) / BT) * p.nt
                          : sh->tiles;

  Schedule sched;
  if constexpr (GROUPED)
    sched.init(T, p, blockIdx.x);
  else
    sched.init_dense(p, blockIdx.x);
  // Programmatic dependent launch: the next grid on the stream may start its
  // CTAs as soon as SMs free up; everything it reads from this grid is read
  // after its own grid_dependency_wait.
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------ weight producer
    // Packed weights are read-only layer data, so they stream before (and
    // regardless of) the wait for the previous grid on the stream.
    if (lane == 0) {
      const uint64_t pol = p.w_reuse ? policy_evict_normal() : policy_evict_first();
      int issued = 0;
      bool skip_first = first_issued;
      int ws = 0;
      uint32_t wph = 0;
      WorkItem wi;
      bool ok = true;
      while (ok && sched.next(wi)) {
        const TileCoord<BT> tc = coords(wi.tile);
        // the blocks of one n-tile's consecutive k-tiles are contiguous
        const uint8_t* src = p.w + tc.e * p.w_expert_stride +
                             ((long long)tc.nt * p.kt + wi.k0) * blk_bytes;
        for (int kt = wi.k0; kt < wi.k1; kt += RW) {
          const int r = min(RW, wi.k1 - kt);
          if (skip_first) {
            // went out at the start of the kernel.  No wait for the slot: the
            // dequant warps may have consumed and released it already, and
            // the release completes the slot's first phase, so a wait for
            // "free" here would wait for its second release instead
            skip_first = false;
          } else {
            if (!mbar_wait(&w_empty[ws], wph ^ 1, abort_flag, p.status, lim,
                           kStatusTimeout | kSiteWeightSlot)) {
              ok = false;
              break;
            }
            if (!qg_check(tc.e >= 0 && tc.e < p.num_experts && tc.nt >= 0 && tc.nt < p.nt &&
                              kt >= 0 && kt + r <= p.kt,
                          p.status)) {
              *abort_flag = 1;   // the slot is not filled: every waiter gives up
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&w_full[ws], r * blk_bytes);
            bulk_load(w_base + ws * p.w_bytes, src + (long long)(kt - wi.k0) * blk_bytes,
                      r * blk_bytes, &w_full[ws], pol);
          }
          ++issued;
          if (++ws == SW) {
            ws = 0;
            wph ^= 1;
          }
        }
      }
      drain_ring(w_full, SW, issued);
    }
  } else if (warp == 3) {
    // ------------------------------------------------ activation producer
    if (lane == 0) {
      prefetch_tmap(&tmap_a);
      const uint64_t pol = policy_evict_last();
      grid_dependency_wait();   // the previous grid may still write the activations
      int issued = 0;
      int xs = 0;
      uint32_t xph = 0;
      WorkItem wi;
      bool ok = true;
      while (ok && sched.next(wi)) {
        const TileCoord<BT> tc = coords(wi.tile);
        for (int kt = wi.k0; kt < wi.k1; kt += RX) {
          if (!mbar_wait(&x_empty[xs], xph ^ 1, abort_flag, p.status, lim, kStatusTimeout | kSiteActSlot)) {
            ok = false;
            break;
          }
          // the RX activation tiles of a slot in one box: [chunk][BT rows][128 bytes]
          mbar_arrive_expect_tx(&x_full[xs], RX * kActUnit);
          tma_load_3d_hint(x_base + xs * p.x_bytes, &tmap_a, &x_full[xs], 0, tc.row0,
                           kt * (MX ? 1 : 2), pol);
          ++issued;
          if (++xs == SX) {
            xs = 0;
            xph ^= 1;
          }
        }
      }
      drain_ring(x_full, SX, issued);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (elect_one()) {
      const uint32_t idesc = MX ? idesc_mxf8f6f4_e4m3(BT) : idesc_f16(FP16 ? 0u : 1u, BT);
      int xs = 0, slot = 0, acc = 0;
      uint32_t xph = 0, aphase = 0, accphase = 0;
      WorkItem wi;
      bool ok = true;
      if constexpr (MX)   // the B scale factors (all 1.0) are written by the epilogue warps
        ok = mbar_wait(sfb_ready, 0, abort_flag, p.status, lim, kStatusTimeout | kSiteScaleFactors);
      while (ok && sched.next(wi)) {
        if (!mbar_wait(&acc_empty[acc], accphase ^ 1, abort_flag, p.status, lim,
                       kStatusTimeout | kSiteAccEmpty))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + kAccCol + acc * BT;
        for (int kt0 = wi.k0; ok && kt0 < wi.k1; kt0 += RX) {
          const int r = min(RX, wi.k1 - kt0);
          if (!mbar_wait(&x_full[xs], xph, abort_flag, p.status, lim, kStatusTimeout | kSiteActFull)) {
            ok = false;
            break;
          }
          const uint32_t sbase = smem_u32(x_base + xs * p.x_bytes);
          for (int i = 0; i < r; ++i) {
            if (!mbar_wait(&a_full[slot], aphase, abort_flag, p.status, lim, kStatusTimeout | kSiteDequantFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t b0 = sbase + i * kActUnit;
            const bool first = (kt0 + i == wi.k0);
            if constexpr (MX) {
              // four K=32 steps over one 128-byte activation row; the scale
              // factor id selects the step's byte of the scale columns
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_ts_mxf8f6f4(d_tmem, tmem_base + slot * kSlotCols + ks * 8,
                                smem_desc_sw128(b0 + ks * 32), idesc_with_sf_ids(idesc, ks, ks),
                                tmem_base + kSfaCol + slot * 4, tmem_base + kSfbCol,
                                (!first || ks > 0) ? 1u : 0u);
            } else {
#pragma unroll
              for (int ks = 0; ks < kTileK / 16; ++ks) {
                const uint32_t boff = (ks >> 2) * (BT * 128) + (ks & 3) * 32;
                mma_ts_f16(d_tmem, tmem_base + slot * kSlotCols + ks * 8,
                           smem_desc_sw128(b0 + boff), idesc, (!first || ks > 0) ? 1u : 0u);
              }
            }
            mma_commit(&a_empty[slot]);
            if (++slot == kASlots) {
              slot = 0;
              aphase ^= 1;
            }
          }
          if (!ok) break;
          mma_commit(&x_empty[xs]);
          if (++xs == SX) {
            xs = 0;
            xph ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
        if (++acc == NACC) {
          acc = 0;
          accphase ^= 1;
        }
      }
      // every MMA this thread issued completes before TMEM is released
      mma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait(drain, 0, &no_abort, nullptr, 100000000ull, 0);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------ dequant
    // Two warps per TMEM lane quadrant; warp group h takes every other unit
    // (h = unit index & 1) and dequantizes all 128 k of its 32 rows.  A warp
    // reads all of its group's units in a weight slot (at most two) into
    // registers as soon as the slot is full and hands the slot back at once;
    // the second unit's shared-memory reads are then off its critical path.
    const int q = warp & 3;             // TMEM lane quadrant
    const int h = (warp - 4) >> 2;      // which units: even (0) or odd (1)
    const int row = q * 32 + lane;      // output feature within the tile
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    constexpr uint32_t magic16 = FP16 ? 0x6400u : 0x4300u;
    int ws = 0;
    uint32_t wph = 0;
    int unit = 0;                       // units of this CTA before the current slot
    WorkItem wi;
    bool ok = true;
    while (ok && sched.next(wi)) {
      for (int kt0 = wi.k0; ok && kt0 < wi.k1; kt0 += RW) {
        const int r = min(RW, wi.k1 - kt0);
        if (!mbar_wait(&w_full[ws], wph, abort_flag, p.status, lim, kStatusTimeout | kSiteWeightFull)) {
          ok = false;
          break;
        }
        const uint8_t* sp = w_base + ws * p.w_bytes;
        const int i0 = ((unit & 1) == h) ? 0 : 1;   // this group's units: i0, i0 + 2
        if constexpr (W8) {
          // 8-bit codes: a unit's row is 128 bytes, so the group's units are
          // read, dequantized and stored one at a time, and the slot goes back
          // once the last of them is in registers
          const int mine = i0 < r ? (r - i0 + 1) / 2 : 0;   // units i0, i0 + 2 below r
          if (mine == 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&w_empty[ws]);
          }
          for (int t = 0; t < mine; ++t) {
            const int i = i0 + 2 * t;
            const uint8_t* bp = sp + i * blk_bytes;   // this unit's packed block
            const uint4* wv = reinterpret_cast<const uint4*>(bp);
            const uint16_t* sv = reinterpret_cast<const uint16_t*>(bp + p.s_off);
            const uint8_t* zv = bp + p.z_off;
            uint32_t sc[4], ze[4];   // per 32 k (a group spans at least 32 k)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int sg = c >> p.sg_shift;
              const uint32_t sbits = sv[sg * kTileN + row];
              const uint32_t zq = p.has_zp ? (uint32_t)zv[sg * kTileN + row] : 128u;
              if constexpr (FP16) {
                sc[c] = sbits * 0x00010001u;
                ze[c] = (0x6400u + zq) * 0x00010001u;   // 1024 + z, a pair
              } else {
                sc[c] = sbits << 16;                      // the bf16 scale as fp32
                ze[c] = __float_as_uint(32768.0f + (float)zq);
              }
            }
            const int g = unit + i;                    // unit index within the CTA
            const int slot = g & (kASlots - 1);
            const uint32_t aphase = (uint32_t)(g / kASlots) & 1u;
            const uint32_t tbase = tmem_base + lane_addr + slot * kSlotCols;
            // the row's 128 codes in two halves of four vectors (16 k each),
            // so that only one half is held in registers
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint4 v8[4];
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) v8[jj] = wv[(q * 8 + 4 * hf + jj) * 32 + lane];
              if (hf == 1 && t == mine - 1) {   // every read of the slot by this warp is done
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[ws]);
              }
              if (hf == 0 && !mbar_wait(&a_empty[slot], aphase ^ 1, abort_flag, p.status, lim,
                                        kStatusTimeout | kSiteTmemSlot)) {
                ok = false;
                break;
              }
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {   // 16 k -> 8 columns each
                const int j = 4 * hf + jj;
                uint32_t out[8];
                dequant_vec8<FP16>(v8[jj], ze[j >> 1], sc[j >> 1], out);
                tmem_st8(tbase + j * 8, out);
              }
            }
            if (!ok) break;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[slot]);
          }
        } else {
          uint4 v[2][4];
          uint32_t scale2[2][4], zero2[2][4], sf[2];
          [[maybe_unused]] uint32_t lo2[2][4];   // F16S: the scales' low terms
  #pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int i = i0 + 2 * t;
            if (i < r) {
              const uint8_t* bp = sp + i * blk_bytes;   // this unit's packed block
              const uint4* wv = reinterpret_cast<const uint4*>(bp);
  #pragma unroll
              for (int j = 0; j < 4; ++j) v[t][j] = wv[(q * 4 + j) * 32 + lane];
              if constexpr (MX) {
                sf[t] = reinterpret_cast<const uint32_t*>(bp + p.s_off)[row];
              } else {
                const uint16_t* sv = reinterpret_cast<const uint16_t*>(bp + p.s_off);
                const uint8_t* zv = bp + p.z_off;
  #pragma unroll
                for (int j = 0; j < 4; ++j) {
                  if constexpr (NV) {   // two 16-k block scales per 32-k chunk
                    scale2[t][j] = (uint32_t)sv[(2 * j) * kTileN + row] * 0x00010001u;
                    zero2[t][j] = (uint32_t)sv[(2 * j + 1) * kTileN + row] * 0x00010001u;
                  } else {
                    const int sg = j >> p.sg_shift;
                    if constexpr (F16S)   // the fp16 scale as two bf16 terms (pairs)
                      split_f16_scale(sv[sg * kTileN + row], scale2[t][j], lo2[t][j]);
                    else
                      scale2[t][j] = (uint32_t)sv[sg * kTileN + row] * 0x00010001u;
                    const uint32_t zq = p.has_zp ? (uint32_t)zv[sg * kTileN + row] : 8u;
                    zero2[t][j] = (magic16 + zq) * 0x00010001u;
                  }
                }
              }
            }
          }
          // every read of the slot by this warp is done (or it holds none of
          // the group's units)
          __syncwarp();
          if (lane == 0) mbar_arrive(&w_empty[ws]);
  #pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int i = i0 + 2 * t;
            if (i >= r) break;
            const int g = unit + i;                    // unit index within the CTA
            const int slot = g & (kASlots - 1);
            const uint32_t aphase = (uint32_t)(g / kASlots) & 1u;
            if (!mbar_wait(&a_empty[slot], aphase ^ 1, abort_flag, p.status, lim,
                           kStatusTimeout | kSiteTmemSlot)) {
              ok = false;
              break;
            }
            if constexpr (MX) {
              // 128 e2m1 codes of this row -> 128 e4m3 bytes (32 columns), and
              // its four e8m0 block scales -> the slot's four scale columns
  #pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t o8[8];
                dequant_vec_mx(v[t][j], o8);
                tmem_st8(tmem_base + lane_addr + slot * kSlotCols + j * 8, o8);
              }
              const uint32_t sf4[4] = {sf[t], sf[t], sf[t], sf[t]};
              tmem_st4(tmem_base + lane_addr + kSfaCol + slot * 4, sf4);
            } else {
              const uint32_t tbase = tmem_base + lane_addr + slot * kSlotCols;
  #pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t out[16];
                if constexpr (NV)
                  dequant_vec_nv<FP16>(v[t][j], scale2[t][j], zero2[t][j], out);
                else if constexpr (F16S)
                  dequant_vec_f16s(v[t][j], zero2[t][j], scale2[t][j], lo2[t][j], out);
                else
                  dequant_vec<FP16>(v[t][j], zero2[t][j], scale2[t][j], out);
                tmem_st16(tbase + j * 16, out);
              }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[slot]);
          }
        }
        unit += r;
        if (++ws == SW) {
          ws = 0;
          wph ^= 1;
        }
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------ epilogue
    grid_dependency_wait();   // workspace and output may still be in use upstream
    const int q = warp & 3;
    const int col = q * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    if (lane == 0) prefetch_tmap(&tmap_c);
    if constexpr (MX) {   // B scale factors: every byte 2^0 (e8m0 127)
      uint32_t ones[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) ones[i] = 0x7F7F7F7Fu;
      tmem_st32(tmem_base + lane_addr + kSfbCol, ones);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfb_ready);
    }
    // Output of 16 rows x this warp's 32 columns: rounded into a per-warp
    // staging buffer (two, used in turn) and written by one tensor store,
    // which drops rows past the end of the output.  A grouped tile's last
    // chunk may end inside the tile (the next rows belong to the next
    // expert); its rows are stored one by one instead.
    uint16_t* stg = epi_stage + q * (2 * 16 * 32);
    int sbuf = 0;
    // The CTA's last item (the end of the kernel's critical path) stages each
    // 16-row chunk in its own 2 KB slot of the then idle activation ring,
    // after the finisher's copied sums, so no chunk waits for an earlier
    // store or reduction to finish reading its buffer.
    uint8_t* last_stage = x_base + BT * 512 + q * (BT / 16) * 2048;
    bool last = false;
    uint32_t staged = 0;   // chunks of the final item staged and not yet stored
    auto emit = [&](const TileCoord<BT>& tc, int m0, const float (&f)[16], float bias) {
      uint16_t o[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float v = f[i];
        if constexpr (MX)   // W4A8: the per-row activation scale multiplies the fp32 sum
          v *= (m0 + i < tc.rows && qg_check(tc.row0 + m0 + i < p.rows, p.status))
                   ? p.a_scale[tc.row0 + m0 + i]
                   : 0.f;
        if constexpr (NV)   // NVFP4: the expert's tensor scale multiplies the fp32 sum
          v *= p.t_scales[tc.e];
        o[i] = to_out<FP16>(v + bias);
      }
      const int valid = tc.rows - m0;
      if constexpr (!FP16) {
        if (p.gated) {
          // Lanes 2j and 2j+1 hold the gate and the up value of output column
          // 64 nt + 16 q + j for the chunk's 16 rows; they swap halves so that
          // the even lane forms rows 0..7 of the gated product, the odd lane
          // rows 8..15.
          const int odd = lane & 1;
          uint32_t pk[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) pk[j] = (uint32_t)o[2 * j] | ((uint32_t)o[2 * j + 1] << 16);
          uint32_t hw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t mine = odd ? pk[4 + j] : pk[j];
            const uint32_t theirs = __shfl_xor_sync(0xffffffffu, odd ? pk[j] : pk[4 + j], 1);
            const uint32_t gw = odd ? theirs : mine, uw = odd ? mine : theirs;
            const float h0 = silu_mul_f32(__uint_as_float(gw << 16), __uint_as_float(uw << 16));
            const float h1 = silu_mul_f32(__uint_as_float(gw & 0xFFFF0000u),
                                          __uint_as_float(uw & 0xFFFF0000u));
            hw[j] = (uint32_t)to_out<false>(h0) | ((uint32_t)to_out<false>(h1) << 16);
          }
          const int r0 = odd * 8, hcol = lane >> 1;
          if (!GROUPED || valid >= 16) {
            uint16_t* sb = last ? reinterpret_cast<uint16_t*>(last_stage + (m0 / 16) * 2048)
                                : stg + sbuf * (16 * 32);   // 16 rows x 16 columns
            if (lane == 0 && !last) bulk_wait_group_read<1>();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              sb[(r0 + 2 * j) * 16 + hcol] = (uint16_t)(hw[j] & 0xFFFF);
              sb[(r0 + 2 * j + 1) * 16 + hcol] = (uint16_t)(hw[j] >> 16);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmap_c, sb, tc.nt * (kTileN / 2) + q * 16, tc.row0 + m0);
              bulk_commit_group();
            }
            sbuf ^= 1;
          } else {
            const int nh = p.n >> 1;
            uint16_t* dst = p.c + (long long)(tc.row0 + m0 + r0) * nh + tc.nt * (kTileN / 2) +
                            q * 16 + hcol;
            const bool in = qg_check(tc.nt * (kTileN / 2) + q * 16 + hcol < nh &&
                                         tc.row0 + m0 + min(valid, 16) <= p.rows,
                                     p.status);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (in && r0 + j < valid)
                dst[(long long)j * nh] = (uint16_t)((hw[j >> 1] >> (16 * (j & 1))) & 0xFFFF);
          }
          return;
        }
      }
      if ((!GROUPED || valid >= 16) && last) {
        // the final item's chunks each have a staging slot of their own:
        // staged now, stored together after the item's last chunk (one
        // proxy fence and one bulk group for the whole item)
        uint16_t* sb = reinterpret_cast<uint16_t*>(last_stage + (m0 / 16) * 2048);
#pragma unroll
        for (int i = 0; i < 16; ++i) sb[i * 32 + lane] = o[i];
        staged |= 1u << (m0 / 16);
      } else if (!GROUPED || valid >= 16) {
        uint16_t* sb = stg + sbuf * (16 * 32);
        if (lane == 0) bulk_wait_group_read<1>();   // the buffer's previous store read it
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 16; ++i) sb[i * 32 + lane] = o[i];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmap_c, sb, tc.nt * kTileN + q * 32, tc.row0 + m0);
          bulk_commit_group();
        }
        sbuf ^= 1;
      } else {
        uint16_t* dst = p.c + (long long)(tc.row0 + m0) * p.n + tc.nt * kTileN + col;
        if (qg_check(tc.nt * kTileN + col < p.n && tc.row0 + m0 + valid <= p.rows, p.status))
          for (int i = 0; i < valid; ++i) dst[(long long)i * p.n] = o[i];
      }
    };
    int acc = 0;
    uint32_t accphase = 0;
    WorkItem wi;
    while (sched.next(wi)) {
      const TileCoord<BT> tc = coords(wi.tile);
      const bool whole = (wi.k0 == 0 && wi.k1 == p.kt);
      bool final_item;
      {
        Schedule peek = sched;
        WorkItem nx;
        final_item = !peek.next(nx);
      }
      if (!mbar_wait(&acc_full[acc], accphase, abort_flag, p.status, lim, kStatusTimeout | kSiteAccFull)) break;
      // after the last item's accumulator is full, every MMA (and so every
      // read of the activation ring) of this CTA has completed
      last = p.last_stage && final_item;
      tc_fence_after();
      const int n = packed_source_col(tc.nt, col, p.n, p.gated);
      const float bias =
          (p.bias && qg_check(tc.e >= 0 && tc.e < p.num_experts && n >= 0 && n < p.n, p.status))
              ? from_out<FP16>(p.bias[(long long)tc.e * p.n + n])
              : 0.f;
      const uint32_t tbase = tmem_base + lane_addr + kAccCol + acc * BT;
      // Split tiles.  A tile's fp32 accumulator is four quadrant blocks of
      // [BT rows][32 columns]: each block is contiguous (one bulk copy for the
      // finisher) and each 8-row slice of it is one 1 KB bulk reduction.
      const int tl = wi.tile - sched.W * sched.G;
      const int u_start = tl * p.kt;
      const int c_first = whole ? 0 : sched.cta_of_unit(u_start);
      const int c_last = whole ? 0 : sched.cta_of_unit(u_start + p.kt - 1);
      const int contributors = (int)(c_last - c_first + 1);
      // split-K bookkeeping of a split tile: its counters and accumulator
      // (atomic mode: one per split tile, at most 2 per CTA; fixed order:
      // two slots per CTA)
      const bool split_ok =
          whole || p.cluster > 1 ||
          qg_check(wi.tile >= 0 && (long long)wi.tile < p.max_tiles && tl >= 0 &&
                       tl < 2 * (int)gridDim.x,
                   p.status);
      int* counter = &p.counters[(long long)wi.tile * 4 + q];
      const bool finisher = !whole && !p.deterministic && c_first == (int)blockIdx.x;
      if (!split_ok) {
        // out-of-range split bookkeeping (checked build): the tile is skipped
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
      } else if (!GROUPED && p.cluster > 1) {
        // Cluster split: the cluster's S CTAs hold the tile's S K slices (this
        // item is the CTA's only one).  16-row chunk mc of quadrant q is unit
        // u = q * BT / 16 + mc, finished by cluster rank u % S: the others
        // send their fp32 partial of it (this lane's feature, 16 rows, 64
        // bytes) into that rank's receive slots, which sums the S slices in
        // rank order (the result does not depend on timing) and stores it.
        constexpr int NCH = BT / 16;
        const int S = p.cluster, sl = (int)(blockIdx.x % (unsigned)S);
        const int nlive = (tc.rows + 15) / 16;
        float* recv = reinterpret_cast<float*>(smem + p.off_recv);   // [u / S][S - 1][32][16]
        if (!cl_waited) {
          cluster_wait();
          cl_waited = true;
        }
        for (int mc = 0; mc < nlive; ++mc) {
          const int u = q * NCH + mc, owner = u % S;
          if (owner == sl) continue;
          uint32_t v[16];
          tmem_ld16_wait(tbase + mc * 16, v);
          const int slot = (u / S) * (S - 1) + (sl < owner ? sl : sl - 1);
          if (!qg_check(owner < S && slot < ((4 * NCH + S - 1) / S) * (S - 1), p.status))
            continue;   // (the owner then gives up its bounded wait)
          const uint32_t dst = map_to_rank(smem_u32(recv + (slot * 32 + lane) * 16), owner);
          const uint32_t bar = map_to_rank(smem_u32(recv_full), owner);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_async_f4(dst + 16 * i,
                        make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])),
                        bar);
        }
        if (mbar_wait(recv_full, 0, abort_flag, p.status, lim, kStatusTimeout | kSiteClusterRecv)) {
#pragma unroll 1
          for (int mc = 0; mc < nlive; ++mc) {
            const int u = q * NCH + mc;
            if (u % S != sl) continue;
            uint32_t v[16];
            tmem_ld16_wait(tbase + mc * 16, v);
            float f[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = 0.f;
            for (int r = 0; r < S; ++r) {
              if (r == sl) {
#pragma unroll
                for (int i = 0; i < 16; ++i) f[i] += __uint_as_float(v[i]);
              } else {
                const int slot = (u / S) * (S - 1) + (r < sl ? r : r - 1);
                const float4* s4 = reinterpret_cast<const float4*>(recv + (slot * 32 + lane) * 16);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float4 x = s4[i];
                  f[4 * i] += x.x;
                  f[4 * i + 1] += x.y;
                  f[4 * i + 2] += x.z;
                  f[4 * i + 3] += x.w;
                }
              }
            }
            emit(tc, mc * 16, f, bias);
          }
        } else {
          // every peer sends, so the slices still arrive: wait (bounded) for
          // them before this CTA's shared memory is released
          volatile int no_abort = 0;
          mbar_wait(recv_full, 0, &no_abort, nullptr, 100000000ull, 0);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
      } else if (whole || (!p.deterministic && !finisher)) {
        // whole tile: output; atomic-mode contributor: add into the tile's
        // accumulator, 8 rows x 32 columns (1 KB) per bulk reduction through
        // the staging buffers.  Only slices holding output rows are added, so
        // rows past the end stay zero in the accumulator.
        float* quad_acc = p.partials + (long long)tl * (BT * kTileN) + q * 32 * BT;
        if (whole) {
          // two 16-row chunks per tensor-memory load (one load latency each;
          // past an odd last chunk the load reads unused columns, inside the
          // allocation: BT / 16 is even from BT = 32 on, and at BT = 16 both
          // accumulators end 32 columns before the allocation does)
          const int nch = min(BT / 16, (tc.rows + 15) / 16);
#pragma unroll 1
          for (int mc = 0; mc < nch; mc += 2) {
            uint32_t v[32];
            tmem_ld32_wait(tbase + mc * 16, v);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (mc + h >= nch) break;
              float f[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[16 * h + i]);
              emit(tc, (mc + h) * 16, f, bias);
            }
          }
        }
#pragma unroll 1
        for (int mc = 0; !whole && mc < BT / 16 && mc * 16 < tc.rows; ++mc) {
          uint32_t v[16];
          tmem_ld16_wait(tbase + mc * 16, v);
          {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (mc * 16 + h * 8 >= tc.rows) break;
              float* sb = last ? reinterpret_cast<float*>(last_stage + mc * 2048 + h * 1024)
                               : reinterpret_cast<float*>(stg + sbuf * (16 * 32));
              if (lane == 0 && !last) bulk_wait_group_read<1>();   // the buffer's previous op read it
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 8; ++i) sb[i * 32 + lane] = __uint_as_float(v[8 * h + i]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                bulk_reduce_add_f32(quad_acc + (mc * 16 + h * 8) * 32, sb, 8 * 32 * 4);
                bulk_commit_group();
              }
              sbuf ^= 1;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&acc_empty[acc]);
          if (!whole) {
            // the reductions complete, then are ordered before the count
            // (async proxy -> generic proxy -> release)
            bulk_wait_group_all();
            fence_proxy_async_global();
            red_release_add_gpu(counter, 1);
          }
        }
      } else if (finisher) {
        // Atomic-mode finisher: the CTA holding the tile's first k-tiles,
        // which (stream-K order) is this CTA's last work item.  Its own
        // partial stays in tensor memory; once the other contributors'
        // counts arrive, their sum is copied in with one bulk copy per
        // quadrant (into the activation ring, idle after the last item's
        // MMAs) or read directly, added, written out, and the accumulator
        // and counter are left at zero for the next launch.
        const bool via_smem = p.fix_smem && final_item;
        float* quad = p.partials + (long long)tl * (BT * kTileN) + q * 32 * BT;
        bool ok = true;
        if (lane == 0) {
          const uint64_t t0 = globaltimer();
          while (ld_acquire_gpu(counter) < contributors - 1) {
            if (*abort_flag || globaltimer() - t0 >= lim) {
              if (!*abort_flag) {
                *abort_flag = 1;
                atomicOr(p.status, kStatusTimeout | kSiteSplitCount);
              }
              ok = false;
              break;
            }
            __nanosleep(64);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
        __syncwarp();   // orders every lane's reads after lane 0's acquire
        const float* sum_col = quad + lane;   // row m of this column at [m * 32]
        if (ok && via_smem) {
          float* fsm = reinterpret_cast<float*>(x_base) + q * 32 * BT;
          if (lane == 0) {
            fence_proxy_async_global();
            mbar_arrive_expect_tx(&fix_bar[q], BT * 128);
            bulk_load(fsm, quad, BT * 128, &fix_bar[q], policy_evict_first());
          }
          __syncwarp();
          ok = mbar_wait(&fix_bar[q], 0, abort_flag, p.status, lim, kStatusTimeout | kSiteSplitCopy);
          if (!ok) {   // never leave the copy writing shared memory the CTA is leaving
            volatile int no_abort = 0;
            mbar_wait(&fix_bar[q], 0, &no_abort, nullptr, 100000000ull, 0);
          }
          sum_col = fsm + lane;
        }
        if (ok) {
#pragma unroll 1
          for (int mc = 0; mc < BT / 16 && mc * 16 < tc.rows; ++mc) {
            uint32_t v[16];
            tmem_ld16_wait(tbase + mc * 16, v);
            const float* s1 = sum_col + mc * 16 * 32;
            float f[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              f[i] = __uint_as_float(v[i]) + (via_smem ? s1[i * 32] : __ldcg(s1 + i * 32));
            emit(tc, mc * 16, f, bias);
          }
          // leave the quadrant's accumulator zeroed (coalesced) and the count reset
          float4* q4 = reinterpret_cast<float4*>(quad);
          for (int i = lane; i < 8 * BT; i += 32) q4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (lane == 0) *counter = 0;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
      } else {
        // fixed-order mode: this CTA's partial to its own slot; the last
        // CTA to arrive for a quadrant sums the slots in CTA order
        const int which = (sched.sk_begin(blockIdx.x) >= u_start) ? 0 : 1;
        float* my_part = p.partials + ((long long)(2 * blockIdx.x + which)) * (BT * kTileN);
#pragma unroll 1
        for (int mc = 0; mc < BT / 16 && mc * 16 < tc.rows; ++mc) {
          uint32_t v[16];
          tmem_ld16_wait(tbase + mc * 16, v);
          float4* dst = reinterpret_cast<float4*>(my_part + col * BT + mc * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        // the warp's partial stores are ordered before lane 0's release add;
        // the acquiring add of the last arrival orders the reads after it
        __syncwarp();
        int old = 0;
        if (lane == 0) old = atomic_add_acq_rel_gpu(counter, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        __syncwarp();
        if (old == contributors - 1) {
          // fixed-order mode: the contributors' partials summed in CTA order,
          // two contributors' loads in flight at a time
          for (int m0 = 0; m0 < tc.rows; m0 += 16) {
            float f[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i] = 0.f;
            for (int cc0 = c_first; cc0 <= c_last; cc0 += 2) {
              float4 v4[2][4];
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const int cc = cc0 + i;
                if (cc <= c_last) {
                  const int which = (sched.sk_begin(cc) >= u_start) ? 0 : 1;
                  const float4* src4 = reinterpret_cast<const float4*>(
                      p.partials + ((long long)(2 * cc + which)) * (BT * kTileN) + col * BT + m0);
#pragma unroll
                  for (int j = 0; j < 4; ++j) v4[i][j] = __ldcg(src4 + j);
                }
              }
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                if (cc0 + i <= c_last) {
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    f[4 * j] += v4[i][j].x;
                    f[4 * j + 1] += v4[i][j].y;
                    f[4 * j + 2] += v4[i][j].z;
                    f[4 * j + 3] += v4[i][j].w;
                  }
                }
              }
            }
            emit(tc, m0, f, bias);
          }
          if (lane == 0) *counter = 0;   // ready for the next launch
        }
      }
      if (staged) {   // the final item's staged chunks
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (uint32_t b = staged; b; b &= b - 1) {
            const int mc = __ffs((int)b) - 1;
            tma_store_2d(&tmap_c, last_stage + mc * 2048, tc.nt * kTileN + q * 32,
                         tc.row0 + mc * 16);
          }
          bulk_commit_group();
        }
        staged = 0;
      }
      if (++acc == NACC) {
        acc = 0;
        accphase ^= 1;
      }
    }
    if (lane == 0) bulk_wait_group_all();   // tensor stores done before the CTA exits
    __syncwarp();
  }

  __syncwarp();
  if (!GROUPED && p.cluster > 1) {
    // No CTA leaves while a peer may still send into its shared memory: the
    // epilogue warps (the last senders) wait for every thread of the cluster
    // to arrive; the others arrive and block in the CTA barrier below, which
    // leaves the issue slots to the epilogue warps meanwhile.
    if (!cl_waited) cluster_wait();
    cluster_arrive();
    if (warp >= 12) cluster_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem_base, 512);
}

// ---------------------------------------------------------------- host side

template <int BT, int FMT, bool GROUPED>
static cudaError_t launch_t(const CUtensorMap& tmap, const CUtensorMap& tmap_c,
                            const W4A16Params& p, int grid, cudaStream_t stream) {
  auto kern = w4a16_kernel<BT, FMT, GROUPED>;
  static int attr_set = 0;   // largest dynamic shared memory size enabled so far
  if (p.smem_bytes > attr_set) {
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
    if (err != cudaSuccess) return err;
    attr_set = p.smem_bytes;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kNumThreads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = p.cluster > 1 ? (unsigned)p.cluster : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (!GROUPED && p.cluster > 1) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, tmap, tmap_c, p);
}

// Clusters of S CTAs of the dense kernel (with smem bytes of dynamic shared
// memory) that fit on the device at once.
template <int BT, int FMT>
static int max_clusters_t(int S, int smem) {
  auto kern = w4a16_kernel<BT, FMT, false>;
  int cap = 0;
  if (cudaDeviceGetAttribute(&cap, cudaDevAttrMaxSharedMemoryPerBlockOptin, 0) != cudaSuccess)
    return 0;
  // the largest size any launch asks for, so a later launch is never refused
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, cap) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(S * 64));
  cfg.blockDim = dim3(kNumThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int FMT>
static int max_clusters_bt(int bt, int S, int smem) {
  switch (bt) {
    case 16: return max_clusters_t<16, FMT>(S, smem);
    case 32: return max_clusters_t<32, FMT>(S, smem);
    case 64: return max_clusters_t<64, FMT>(S, smem);
    case 128: return max_clusters_t<128, FMT>(S, smem);
    default: return 0;
  }
}

int w4a16_max_clusters(int bt, int fmt, int S, int smem) {
  // one GPU model per process (the library runs on sm_103 only)
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, int> cache;
  const auto key = std::make_tuple(bt, fmt, S, smem);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int n = 0;
  switch (fmt) {
    case 0: n = max_clusters_bt<0>(bt, S, smem); break;
    case 1: n = max_clusters_bt<1>(bt, S, smem); break;
    case 2: n = max_clusters_bt<2>(bt, S, smem); break;
    case 3: n = max_clusters_bt<3>(bt, S, smem); break;
    case 4: n = max_clusters_bt<4>(bt, S, smem); break;
    case 5: n = max_clusters_bt<5>(bt, S, smem); break;
    case 6: n = max_clusters_bt<6>(bt, S, smem); break;
    case 7: n = max_clusters_bt<7>(bt, S, smem); break;
    default: n = 0;
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = n;
  return n;
}

template <int FMT, bool GROUPED>
static cudaError_t launch_bt(const CUtensorMap& tmap, const CUtensorMap& tmap_c,
                             const W4A16Params& p, int bt, int grid, cudaStream_t stream) {
  switch (bt) {
    case 16: return launch_t<16, FMT, GROUPED>(tmap, tmap_c, p, grid, stream);
    case 32: return launch_t<32, FMT, GROUPED>(tmap, tmap_c, p, grid, stream);
    case 64: return launch_t<64, FMT, GROUPED>(tmap, tmap_c, p, grid, stream);
    case 128: return launch_t<128, FMT, GROUPED>(tmap, tmap_c, p, grid, stream);
    case 256:
      if constexpr (FMT == 0 || FMT == 1)
        return launch_t<256, FMT, GROUPED>(tmap, tmap_c, p, grid, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_w4a16(const CUtensorMap& tmap_a, const CUtensorMap& tmap_c,
                         const W4A16Params& p, int block_tok, int fmt, bool grouped, int grid,
                         cudaStream_t stream) {
  switch (fmt) {
    case 0: return grouped ? launch_bt<0, true>(tmap_a, tmap_c, p, block_tok, grid, stream)
                           : launch_bt<0, false>(tmap_a, tmap_c, p, block_tok, grid, stream);
    case 1: return grouped ? launch_bt<1, true>(tmap_a, tmap_c, p, block_tok, grid, stream)
                           : launch_bt<1, false>(tmap_a, tmap_c, p, block_tok, grid, stream);
    case 2: return grouped ? launch_bt<2, true>(tmap_a, tmap_c, p, block_tok, grid, stream)
                           : launch_bt<2, false>(tmap_a, tmap_c, p, block_tok, grid, stream);
    case 3: return grouped ? launch_bt<3, true>(tmap_a, tmap_c, p, block_tok, grid, stream)
                           : launch_bt<3, false>(tmap_a, tmap_c, p, block_tok, grid, stream);
    case 4: return grouped ? launch_bt<4, true>(tmap_a, tmap_c, p, block_tok, grid, stream)
                           : launch_bt<4, false>(tmap_a, tmap_c, p, block_tok, grid, stream);
    case 5: return grouped ? launch_bt<5, true>(tmap_a, tmap_c, p, block_tok, grid, stream)
                           : launch_bt<5, false>(tmap_a, tmap_c, p, block_tok, grid, stream);
    case 6: return grouped ? launch_bt<6, true>(tmap_a, tmap_c, p, block_tok, grid, stream)
                           : launch_bt<6, false>(tmap_a, tmap_c, p, block_tok, grid, stream);
    case 7: return grouped ? launch_bt<7, true>(tmap_a, tmap_c, p, block_tok, grid, stream)
                           : launch_bt<7, false>(tmap_a, tmap_c, p, block_tok, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

// ------------------------------------------------------------ debug dequant

// out[k, n] = the value the GEMM kernel feeds the tensor core for W^[k, n]
// (NVFP4: e2m1 x block scale; the tensor scale is applied to the fp32 sum).
// F16S: bf16 output from fp16 scales.
template <bool FP16, bool NV, bool F16S>
__global__ void debug_dequant_kernel(const uint8_t* packed, uint16_t* out, int n, int k,
                                     int group, int has_zp, int gated) {
  const int KT = k / kTileK;
  const long long vec = (long long)blockIdx.x * blockDim.x + threadIdx.x;   // one 16-byte vector
  const long long total = (long long)(n / kTileN) * KT * 512;
  if (vec >= total) return;
  const long long blk = vec / 512;
  const int v = (int)(vec % 512);
  const int nt = (int)(blk / KT), kt = (int)(blk % KT);
  const int t = v & 31, j = (v >> 5) & 3, q = v >> 7;
  const int row = q * 32 + t;
  const int st = group < kTileK ? kTileK / group : 1;
  const int sg = group < kTileK ? (32 * j) / group : 0;
  const uint8_t* bp = packed + blk * packed_block_bytes(false, st, has_zp != 0);
  const uint4 wv = reinterpret_cast<const uint4*>(bp)[v];
  const uint32_t sbits = reinterpret_cast<const uint16_t*>(bp + kTileBytes)[sg * kTileN + row];
  const uint32_t zq =
      has_zp ? (uint32_t)(bp + kTileBytes + packed_scale_bytes(false, st))[sg * kTileN + row] : 8u;
  constexpr uint32_t magic16 = FP16 ? 0x6400u : 0x4300u;
  uint32_t o[16];
  if constexpr (NV) {   // two 16-k block scales for the vector's 32 k
    const uint16_t* sv = reinterpret_cast<const uint16_t*>(bp + kTileBytes);
    dequant_vec_nv<FP16>(wv, (uint32_t)sv[(2 * j) * kTileN + row] * 0x00010001u,
                         (uint32_t)sv[(2 * j + 1) * kTileN + row] * 0x00010001u, o);
  } else if constexpr (F16S) {
    uint32_t hi2, lo2;
    split_f16_scale((uint16_t)sbits, hi2, lo2);
    dequant_vec_f16s(wv, (magic16 + zq) * 0x00010001u, hi2, lo2, o);
  } else {
    dequant_vec<FP16>(wv, (magic16 + zq) * 0x00010001u, sbits * 0x00010001u, o);
  }
  const int nn = packed_source_col(nt, row, n, gated);
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const int kk = kt * kTileK + j * 32 + 2 * c;
    out[(long long)kk * n + nn] = (uint16_t)(o[c] & 0xFFFF);
    out[(long long)(kk + 1) * n + nn] = (uint16_t)(o[c] >> 16);
  }
}

// W8A16: the 8-bit blocks' 1024 vectors (16 k of one row each).
template <bool FP16>
__global__ void debug_dequant8_kernel(const uint8_t* packed, uint16_t* out, int n, int k,
                                      int group, int has_zp, int gated) {
  const int KT = k / kTileK;
  const long long vec = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)(n / kTileN) * KT * 1024;
  if (vec >= total) return;
  const long long blk = vec / 1024;
  const int v = (int)(vec % 1024);
  const int nt = (int)(blk / KT), kt = (int)(blk % KT);
  const int t = v & 31, j = (v >> 5) & 7, q = v >> 8;
  const int row = q * 32 + t;
  const int st = group < kTileK ? kTileK / group : 1;
  const int sg = group < kTileK ? (16 * j) / group : 0;
  const uint8_t* bp = packed + blk * packed_block_bytes(false, st, has_zp != 0, true);
  const uint4 wv = reinterpret_cast<const uint4*>(bp)[v];
  const uint32_t sbits =
      reinterpret_cast<const uint16_t*>(bp + packed_code_bytes(true))[sg * kTileN + row];
  const uint32_t zq =
      has_zp ? (uint32_t)(bp + packed_code_bytes(true) + packed_scale_bytes(false, st))[sg * kTileN + row]
             : 128u;
  uint32_t o[8];
  if constexpr (FP16)
    dequant_vec8<true>(wv, (0x6400u + zq) * 0x00010001u, sbits * 0x00010001u, o);
  else
    dequant_vec8<false>(wv, __float_as_uint(32768.0f + (float)zq), sbits << 16, o);
  const int nn = packed_source_col(nt, row, n, gated);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int kk = kt * kTileK + j * 16 + 2 * c;
    out[(long long)kk * n + nn] = (uint16_t)(o[c] & 0xFFFF);
    out[(long long)(kk + 1) * n + nn] = (uint16_t)(o[c] >> 16);
  }
}

cudaError_t launch_debug_dequant(const uint8_t* packed, uint16_t* out, int64_t n, int64_t k,
                                 int group, int has_zp, bool fp16, bool nv, bool f16s,
                                 bool w8, int gated, cudaStream_t stream) {
  const int threads = 256;
  if (w8) {
    const long long total8 = (n / kTileN) * (k / kTileK) * 1024;
    auto kern8 = fp16 ? debug_dequant8_kernel<true> : debug_dequant8_kernel<false>;
    kern8<<<(unsigned)((total8 + threads - 1) / threads), threads, 0, stream>>>(
        packed, out, (int)n, (int)k, group, has_zp, gated);
    return cudaGetLastError();
  }
  const long long total = (n / kTileN) * (k / kTileK) * 512;
  const unsigned blocks = (unsigned)((total + threads - 1) / threads);
  auto kern = fp16   ? (nv ? debug_dequant_kernel<true, true, false>
                           : debug_dequant_kernel<true, false, false>)
              : nv   ? debug_dequant_kernel<false, true, false>
              : f16s ? debug_dequant_kernel<false, false, true>
                     : debug_dequant_kernel<false, false, false>;
  kern<<<blocks, threads, 0, stream>>>(packed, out, (int)n, (int)k, group, has_zp, gated);
  return cudaGetLastError();
}

// out[k, n] = the e4m3 byte the W4A8 kernel writes to tensor memory for the
// code of W[k, n] (the e8m0 block scale is applied by the MMA, not here).
__global__ void debug_mx_codes_kernel(const uint8_t* w, uint8_t* out, int n, int k, int gated) {
  const int KT = k / kTileK;
  const long long vec = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)(n / kTileN) * KT * 512;
  if (vec >= total) return;
  const long long blk = vec / 512;
  const int v = (int)(vec % 512);
  const int nt = (int)(blk / KT), kt = (int)(blk % KT);
  const int t = v & 31, j = (v >> 5) & 3, q = v >> 7;
  uint32_t o[8];
  dequant_vec_mx(reinterpret_cast<const uint4*>(w + blk * packed_block_bytes(true, 1, false))[v],
                 o);
  const int nn = packed_source_col(nt, q * 32 + t, n, gated);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const int kk = kt * kTileK + j * 32 + c;
    out[(long long)kk * n + nn] = (uint8_t)((o[c >> 2] >> (8 * (c & 3))) & 0xFF);
  }
}

cudaError_t launch_debug_mx_codes(const uint8_t* w, uint8_t* out_kn, int64_t n, int64_t k,
                                  int gated, cudaStream_t stream) {
  const long long total = (n / kTileN) * (k / kTileK) * 512;
  debug_mx_codes_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(w, out_kn, (int)n,
                                                                           (int)k, gated);
  return cudaGetLastError();
}

}  // namespace qg
