// W4A16 GEMM for sm_103a: C[M, N] = A[M, K] . W^[K, N], W^ = adt((q - z) * s).
//
// The Humming pages assemble their kernels from scheduling, data movement,
// dequantization/scaling, tensor-core compute and output processing
// (kinachrichten.com, "Kompilierzeiten und geraetespezifisches Tuning"), with
// a TMA + UMMA pipeline for larger batches and a multi-stage cp.async + MMA
// pipeline for small ones (same article, section "Kompilierzeiten...",
// paragraph on small vs larger batch sizes).  This kernel is the B300 design
// of those five components, one kernel for every M:
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
//             stores; or an fp32 partial tile plus a fixed-order reduction by
//             the last-arriving CTA when a tile's K range was split.
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

#include "internal.h"
#include "ptx.cuh"

namespace qg {

namespace {

struct WorkItem {
  int tile;
  int k0, k1;
};

// Whole tiles round-robin (waves), then an even split of the remaining tiles'
// K-tiles ("units") across the first Gs = min(G, U) CTAs, so that every CTA
// taking part in the split owns at least one unit; the CTAs that share a tile
// are then exactly cta_of_unit(first unit) .. cta_of_unit(last unit).
struct Schedule {
  long long T;     // tiles
  int KT;          // k-tiles per tile
  int G, c;        // grid size, this CTA
  long long W;     // full waves of whole tiles
  long long U;     // stream-K units
  long long Gs;    // CTAs sharing the stream-K units
  long long it, u, u_end;

  __device__ void init(long long T_, int KT_, int G_, int c_) {
    T = T_;
    KT = KT_;
    G = G_;
    c = c_;
    W = T / G;
    U = (T - W * G) * KT;
    Gs = U < G ? U : G;
    it = 0;
    if (c < Gs) {
      u = sk_begin(c);
      u_end = sk_begin(c + 1);
    } else {
      u = u_end = 0;
    }
  }
  __device__ long long sk_begin(long long cta) const { return (cta * U) / Gs; }
  // CTA whose unit range holds unit uu.
  __device__ long long cta_of_unit(long long uu) const { return ((uu + 1) * Gs - 1) / U; }

  __device__ bool next(WorkItem& wi) {
    if (it < W) {
      wi.tile = (int)(c + it * G);
      wi.k0 = 0;
      wi.k1 = KT;
      ++it;
      return true;
    }
    if (u >= u_end) return false;
    long long tl = u / KT;
    int k0 = (int)(u % KT);
    long long seg_end = min((tl + 1) * KT, u_end);
    wi.tile = (int)(W * G + tl);
    wi.k0 = k0;
    wi.k1 = k0 + (int)(seg_end - u);
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

// Fire-and-forget fp32 vector reduction into global memory (performed at L2).
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a),
               "f"(b), "f"(c), "f"(d)
               : "memory");
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
// activations with per-row fp32 scales, block-scaled MMA, bf16 output).
//
// A pipeline stage holds up to R = units_per_stage(BT) consecutive k-tiles
// ("units") of one output tile, so that each stage is filled by few, large
// copies: one bulk copy of R weight blocks, one of their scales (and zero
// points), and one three-dimensional TMA box holding the R activation tiles.
template <int BT, int FMT, bool GROUPED>
__global__ void __launch_bounds__(kNumThreads, 1)
    w4a16_kernel(const __grid_constant__ CUtensorMap tmap_a, const W4A16Params p) {
  constexpr bool FP16 = FMT == 1;
  constexpr bool MX = FMT == 2;
  constexpr int R = units_per_stage(BT);
  // tensor-memory columns: dequantized weight slots, then (MX) the A and B
  // scale factors, accumulators from column 256
  constexpr int kSlotCols = MX ? 32 : kASlotCols;
  constexpr uint32_t kSfaCol = 128, kSfbCol = 160, kAccCol = 256;
  constexpr uint32_t kActUnit = BT * kTileK * (MX ? 1 : 2);   // bytes of one unit's activations

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled operand tiles
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int S = p.stages;
  uint8_t* stage_base = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * p.stage_bytes);
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* a_full = empty + S;
  uint64_t* a_empty = a_full + kASlots;
  uint64_t* acc_full = a_empty + kASlots;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* sfb_ready = drain + 1;
  SharedState* sh = reinterpret_cast<SharedState*>(sfb_ready + 1);
  int* mt_prefix = reinterpret_cast<int*>(sh + 1);     // grouped: m-tile prefix [E+1]
  int* offs = mt_prefix + (GROUPED ? (p.num_experts + 1) : 0);   // grouped: offsets [E+1]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sh->abort_flag;
  const uint64_t lim = p.wait_limit_ns;

  auto coords = [&](int tile) {
    TileCoord<BT> tc;
    const int mtg = tile / p.nt;
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

  uint64_t pol_stream = 0, pol_keep = 0;   // L2 policies (set by thread 0)
  const uint32_t blk_bytes = p.block_bytes;   // packed block: codes, scales, zero points

  // ---- producer state (thread 0): one stage = up to R units of one work item
  Schedule psched;
  WorkItem pwi{0, 0, 0};
  int pkt = 0, pr = 0;             // first k-tile and unit count of the current stage
  bool phave = false;
  int pstage = 0;
  uint32_t pphase = 0;
  long long issued = 0;            // stages issued
  auto pnext = [&]() -> bool {     // advance to the next stage; false when none is left
    if (phave && pkt + pr < pwi.k1) {
      pkt += pr;
    } else {
      if (!psched.next(pwi)) return false;
      phave = true;
      pkt = pwi.k0;
    }
    pr = min(R, pwi.k1 - pkt);
    return true;
  };
  // weights, scales and zero points of the current stage: read-only layer
  // data, so they may be requested before the previous grid has finished
  auto issue_weights = [&]() {
    const TileCoord<BT> tc = coords(pwi.tile);
    uint8_t* sp = stage_base + pstage * p.stage_bytes;
    const long long blk = (long long)tc.nt * p.kt + pkt;
    // the pr packed blocks of one n-tile's consecutive k-tiles are contiguous
    mbar_arrive_expect_tx(&full[pstage], R * kActUnit + pr * blk_bytes);
    bulk_load(sp + p.off_w, p.w + tc.e * p.w_expert_stride + blk * blk_bytes, pr * blk_bytes,
              &full[pstage], pol_stream);
  };
  // the R activation tiles of a stage in one box: [chunk][BT rows][128 bytes]
  auto issue_act = [&](int stage, int tile, int kt) {
    const TileCoord<BT> tc = coords(tile);
    tma_load_3d_hint(stage_base + stage * p.stage_bytes, &tmap_a, &full[stage], 0, tc.row0,
                     kt * (MX ? 1 : 2), pol_keep);
  };
  auto advance_pstage = [&]() {
    ++issued;
    if (++pstage == S) {
      pstage = 0;
      pphase ^= 1;
    }
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kASlots; ++i) {
      mbar_init(&a_full[i], 4);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(drain, 1);
    mbar_init(sfb_ready, 4);
    sh->abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmap_a);
    pol_stream = policy_evict_first();
    pol_keep = policy_evict_last();
  }
  if (warp == 2) {
    tmem_alloc(&sh->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 3) {
    if constexpr (GROUPED) {
      // m-tile prefix over experts, from the device-side offsets (written by
      // the previous grid on the stream, so wait for it first)
      grid_dependency_wait();
      const int E = p.num_experts;
      for (int i = lane; i <= E; i += 32) offs[i] = min(max(p.expert_offsets[i], 0), p.rows);
      __syncwarp();
      if (lane == 0) {
        // offsets are caller data: clamp to [0, rows] and make them monotone so
        // that no tile reaches outside the row range
        offs[0] = 0;
        for (int e = 1; e <= E; ++e) offs[e] = max(offs[e], offs[e - 1]);
        int acc = 0;
        mt_prefix[0] = 0;
        for (int e = 0; e < E; ++e) {
          acc += (offs[e + 1] - offs[e] + BT - 1) / BT;
          mt_prefix[e + 1] = acc;
        }
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
  // Start-up barrier.  For a dense GEMM the producer warp only arrives (it
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
  const uint32_t tmem_base = (!GROUPED && warp == 0) ? 0u : sh->tmem_base;
  const long long T = (!GROUPED && warp == 0)
                          ? (long long)((p.rows + BT - 1) / BT) * p.nt
                          : sh->tiles;

  Schedule sched;
  sched.init(T, p.kt, gridDim.x, blockIdx.x);

  // Programmatic dependent launch: the next grid on the stream may start its
  // CTAs as soon as SMs free up; everything it reads from this grid is read
  // after its own grid_dependency_wait.
  grid_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      psched.init(T, p.kt, gridDim.x, blockIdx.x);
      // the first S stages' weights go out before waiting for the previous
      // grid on the stream (which may still write this GEMM's activations or
      // workspace); their activation boxes follow the wait
      int pre = 0;
      int pre_tile[16], pre_kt[16];
      while (pre < S && pnext()) {
        issue_weights();
        pre_tile[pre] = pwi.tile;
        pre_kt[pre] = pkt;
        ++pre;
        advance_pstage();
      }
      grid_dependency_wait();
      for (int i = 0; i < pre; ++i) issue_act(i, pre_tile[i], pre_kt[i]);
      while (pnext()) {
        if (!mbar_wait(&empty[pstage], pphase ^ 1, abort_flag, p.status, lim, kStatusTimeout))
          break;
        issue_weights();
        issue_act(pstage, pwi.tile, pkt);
        advance_pstage();
      }
      // drain: never leave a copy in flight into shared memory we are leaving
      for (int st = 0; st < S && st < issued; ++st) {
        long long last = st + ((issued - 1 - st) / S) * S;
        uint32_t par = (uint32_t)((last / S) & 1);
        volatile int no_abort = 0;
        mbar_wait(&full[st], par, &no_abort, nullptr, 100000000ull, 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (elect_one()) {
      const uint32_t idesc = MX ? idesc_mxf8f6f4_e4m3(BT) : idesc_f16(FP16 ? 0u : 1u, BT);
      int stage = 0, slot = 0, acc = 0;
      uint32_t phase = 0, aphase = 0, accphase = 0;
      WorkItem wi;
      bool ok = true;
      if constexpr (MX)   // the B scale factors (all 1.0) are written by the epilogue warps
        ok = mbar_wait(sfb_ready, 0, abort_flag, p.status, lim, kStatusTimeout);
      while (ok && sched.next(wi)) {
        if (!mbar_wait(&acc_empty[acc], accphase ^ 1, abort_flag, p.status, lim,
                       kStatusTimeout))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + kAccCol + acc * BT;
        for (int kt0 = wi.k0; ok && kt0 < wi.k1; kt0 += R) {
          const int r = min(R, wi.k1 - kt0);
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status, lim, kStatusTimeout)) {
            ok = false;
            break;
          }
          const uint32_t sbase = smem_u32(stage_base + stage * p.stage_bytes);
          for (int i = 0; i < r; ++i) {
            if (!mbar_wait(&a_full[slot], aphase, abort_flag, p.status, lim, kStatusTimeout)) {
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
          mma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&acc_full[acc]);
        if (++acc == 2) {
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
    // (h = unit index & 1) and dequantizes all 128 k of its 32 rows.
    const int q = warp & 3;             // TMEM lane quadrant
    const int h = (warp - 4) >> 2;      // which units: even (0) or odd (1)
    const int row = q * 32 + lane;      // output feature within the tile
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    constexpr uint32_t magic16 = FP16 ? 0x6400u : 0x4300u;
    int stage = 0, slot = 0;
    uint32_t phase = 0, aphase = 0;
    long long unit = 0;
    WorkItem wi;
    bool ok = true;
    while (ok && sched.next(wi)) {
      for (int kt0 = wi.k0; ok && kt0 < wi.k1; kt0 += R) {
        const int r = min(R, wi.k1 - kt0);
        const uint8_t* sp = stage_base + stage * p.stage_bytes;
        for (int i = 0; i < r; ++i, ++unit) {
          if ((unit & 1) == h) {
            if (!mbar_wait(&full[stage], phase, abort_flag, p.status, lim, kStatusTimeout) ||
                !mbar_wait(&a_empty[slot], aphase ^ 1, abort_flag, p.status, lim,
                           kStatusTimeout)) {
              ok = false;
              break;
            }
            const uint8_t* bp = sp + p.off_w + i * blk_bytes;   // this unit's packed block
            const uint4* wv = reinterpret_cast<const uint4*>(bp);
            if constexpr (MX) {
              // 128 e2m1 codes of this row -> 128 e4m3 bytes (32 columns), and
              // its four e8m0 block scales -> the slot's four scale columns
              uint4 v[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) v[j] = wv[(q * 4 + j) * 32 + lane];
              const uint32_t sf =
                  reinterpret_cast<const uint32_t*>(bp + p.s_off)[row];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t o8[8];
                dequant_vec_mx(v[j], o8);
                tmem_st8(tmem_base + lane_addr + slot * kSlotCols + j * 8, o8);
              }
              const uint32_t sf4[4] = {sf, sf, sf, sf};
              tmem_st4(tmem_base + lane_addr + kSfaCol + slot * 4, sf4);
            } else {
              const uint16_t* sv = reinterpret_cast<const uint16_t*>(bp + p.s_off);
              const uint8_t* zv = bp + p.z_off;
              // every shared-memory read of the unit first, then the arithmetic
              uint4 v[4];
              uint32_t scale2[4], zero2[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) v[j] = wv[(q * 4 + j) * 32 + lane];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int sg = j >> p.sg_shift;
                scale2[j] = (uint32_t)sv[sg * kTileN + row] * 0x00010001u;
                const uint32_t zq = p.has_zp ? (uint32_t)zv[sg * kTileN + row] : 8u;
                zero2[j] = (magic16 + zq) * 0x00010001u;
              }
              const uint32_t tbase = tmem_base + lane_addr + slot * kSlotCols;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t out[16];
                dequant_vec<FP16>(v[j], zero2[j], scale2[j], out);
                tmem_st16(tbase + j * 16, out);
              }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[slot]);
          }
          if (++slot == kASlots) {
            slot = 0;
            aphase ^= 1;
          }
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------ epilogue
    grid_dependency_wait();   // workspace and output may still be in use upstream
    const int q = warp & 3;
    const int col = q * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
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
    int acc = 0;
    uint32_t accphase = 0;
    WorkItem wi;
    while (sched.next(wi)) {
      const TileCoord<BT> tc = coords(wi.tile);
      const bool whole = (wi.k0 == 0 && wi.k1 == p.kt);
      if (!mbar_wait(&acc_full[acc], accphase, abort_flag, p.status, lim, kStatusTimeout)) break;
      tc_fence_after();
      const int n = tc.nt * kTileN + col;
      float bias = 0.f;
      if (p.bias) bias = from_out<FP16>(p.bias[(long long)tc.e * p.n + n]);
      const uint32_t tbase = tmem_base + lane_addr + kAccCol + acc * BT;
      // W4A8: the per-row activation scale multiplies the fp32 accumulator
      auto row_scale = [&](int m) -> float {
        if constexpr (MX) return p.a_scale[tc.row0 + m];
        else return 1.f;
      };
      // partial slot of this CTA for this segment (split tiles only)
      const long long tl = wi.tile - sched.W * sched.G;
      const long long u_start = tl * p.kt;
      // split tiles: fixed-order mode writes this CTA's partial to its own
      // slot; atomic mode adds it into the tile's accumulator
      float* my_part = nullptr;
      if (!whole) {
        if (p.deterministic) {
          const int which = (sched.sk_begin(blockIdx.x) >= u_start) ? 0 : 1;
          my_part = p.partials + ((long long)(2 * blockIdx.x + which)) * (BT * kTileN);
        } else {
          my_part = p.partials + tl * (BT * kTileN);
        }
      }
#pragma unroll 1
      for (int mc = 0; mc < BT / 16; ++mc) {
        uint32_t v[16];
        tmem_ld16_wait(tbase + mc * 16, v);
        if (whole) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int m = mc * 16 + i;
            if (m < tc.rows)
              p.c[(long long)(tc.row0 + m) * p.n + n] =
                  to_out<FP16>(__uint_as_float(v[i]) * row_scale(m) + bias);
          }
        } else if (p.deterministic) {
          // partial tile, column-major [col][BT]: this thread's column is contiguous
          float4* dst = reinterpret_cast<float4*>(my_part + col * BT + mc * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        } else {
          float* dst = my_part + col * BT + mc * 16;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            red_add_v4(dst + 4 * i, __uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                       __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        accphase ^= 1;
      }
      if (!whole) {
        // Split-K fixup, per 32-column quadrant, by the warp of the last CTA
        // to arrive for this quadrant of the tile.  The warp's partial stores
        // (or reductions) are ordered before lane 0's release add; the
        // acquiring add of the last arrival orders the reads after it.
        const long long c_first = sched.cta_of_unit(u_start);
        const long long c_last = sched.cta_of_unit(u_start + p.kt - 1);
        const int contributors = (int)(c_last - c_first + 1);
        int* counter = &p.counters[(long long)wi.tile * 4 + q];
        __syncwarp();
        int old = 0;
        if (lane == 0) old = atomic_add_acq_rel_gpu(counter, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        __syncwarp();   // orders every lane's reads after lane 0's acquire
        if (old == contributors - 1 && !p.deterministic) {
          // atomic mode: the accumulator holds the sum; read it (32 rows per
          // pass, all loads issued before use), write the output, and leave
          // the accumulator zeroed for the next launch
          const float4* src4 = reinterpret_cast<const float4*>(my_part + col * BT);
          float4* z4 = reinterpret_cast<float4*>(my_part + col * BT);
          for (int m0 = 0; m0 < tc.rows; m0 += 32) {
            float4 a4[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if (m0 + 4 * j < BT) a4[j] = __ldcg(src4 + m0 / 4 + j);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (m0 + 4 * j < BT) {
                z4[m0 / 4 + j] = make_float4(0.f, 0.f, 0.f, 0.f);
                const float* af = reinterpret_cast<const float*>(&a4[j]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int m = m0 + 4 * j + i;
                  if (m < tc.rows)
                    p.c[(long long)(tc.row0 + m) * p.n + n] =
                        to_out<FP16>(af[i] * row_scale(m) + bias);
                }
              }
            }
          }
          // rows past tc.rows hold what the MMA computed for the tile's padding
          // rows (zero fill or the next expert's tokens): clear them as well
          for (int m0 = ((tc.rows + 31) / 32) * 32; m0 < BT; m0 += 4)
            z4[m0 / 4] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (lane == 0) *counter = 0;   // ready for the next launch
        } else if (old == contributors - 1) {
          // fixed-order mode, 8 rows per pass; up to 4 contributors' partials
          // are loaded before any is added, then summed in CTA order
          for (int m0 = 0; m0 < tc.rows; m0 += 8) {
            float4 acc4[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
            for (long long cc0 = c_first; cc0 <= c_last; cc0 += 4) {
              float4 v4[4][2];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const long long cc = cc0 + i;
                if (cc <= c_last) {
                  const int which = (sched.sk_begin(cc) >= u_start) ? 0 : 1;
                  const float4* src4 = reinterpret_cast<const float4*>(
                      p.partials + ((long long)(2 * cc + which)) * (BT * kTileN) + col * BT + m0);
                  v4[i][0] = __ldcg(src4);
                  v4[i][1] = __ldcg(src4 + 1);
                }
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                if (cc0 + i <= c_last) {
#pragma unroll
                  for (int j = 0; j < 2; ++j) {
                    acc4[j].x += v4[i][j].x;
                    acc4[j].y += v4[i][j].y;
                    acc4[j].z += v4[i][j].z;
                    acc4[j].w += v4[i][j].w;
                  }
                }
              }
            }
            const float* accf = reinterpret_cast<const float*>(acc4);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (m0 + i < tc.rows)
                p.c[(long long)(tc.row0 + m0 + i) * p.n + n] =
                    to_out<FP16>(accf[i] * row_scale(m0 + i) + bias);
            }
          }
          if (lane == 0) *counter = 0;   // ready for the next launch
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem_base, 512);
}

// ---------------------------------------------------------------- host side

template <int BT, int FMT, bool GROUPED>
static cudaError_t launch_t(const CUtensorMap& tmap, const W4A16Params& p, int grid,
                            cudaStream_t stream) {
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmap, p);
}

template <int FMT, bool GROUPED>
static cudaError_t launch_bt(const CUtensorMap& tmap, const W4A16Params& p, int bt, int grid,
                             cudaStream_t stream) {
  switch (bt) {
    case 16: return launch_t<16, FMT, GROUPED>(tmap, p, grid, stream);
    case 32: return launch_t<32, FMT, GROUPED>(tmap, p, grid, stream);
    case 64: return launch_t<64, FMT, GROUPED>(tmap, p, grid, stream);
    case 128: return launch_t<128, FMT, GROUPED>(tmap, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_w4a16(const CUtensorMap& tmap_a, const W4A16Params& p, int block_tok,
                         int fmt, bool grouped, int grid, cudaStream_t stream) {
  switch (fmt) {
    case 0: return grouped ? launch_bt<0, true>(tmap_a, p, block_tok, grid, stream)
                           : launch_bt<0, false>(tmap_a, p, block_tok, grid, stream);
    case 1: return grouped ? launch_bt<1, true>(tmap_a, p, block_tok, grid, stream)
                           : launch_bt<1, false>(tmap_a, p, block_tok, grid, stream);
    case 2: return grouped ? launch_bt<2, true>(tmap_a, p, block_tok, grid, stream)
                           : launch_bt<2, false>(tmap_a, p, block_tok, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

// ------------------------------------------------------------ debug dequant

// out[k, n] = the value the GEMM kernel feeds the tensor core for W^[k, n].
template <bool FP16>
__global__ void debug_dequant_kernel(const uint8_t* packed, uint16_t* out, int n, int k,
                                     int group, int has_zp) {
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
  dequant_vec<FP16>(wv, (magic16 + zq) * 0x00010001u, sbits * 0x00010001u, o);
  const int nn = nt * kTileN + row;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const int kk = kt * kTileK + j * 32 + 2 * c;
    out[(long long)kk * n + nn] = (uint16_t)(o[c] & 0xFFFF);
    out[(long long)(kk + 1) * n + nn] = (uint16_t)(o[c] >> 16);
  }
}

cudaError_t launch_debug_dequant(const uint8_t* packed, uint16_t* out, int64_t n, int64_t k,
                                 int group, int has_zp, bool fp16, cudaStream_t stream) {
  const long long total = (n / kTileN) * (k / kTileK) * 512;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  if (fp16)
    debug_dequant_kernel<true><<<blocks, threads, 0, stream>>>(packed, out, (int)n, (int)k,
                                                                group, has_zp);
  else
    debug_dequant_kernel<false><<<blocks, threads, 0, stream>>>(packed, out, (int)n, (int)k,
                                                                 group, has_zp);
  return cudaGetLastError();
}

// out[k, n] = the e4m3 byte the W4A8 kernel writes to tensor memory for the
// code of W[k, n] (the e8m0 block scale is applied by the MMA, not here).
__global__ void debug_mx_codes_kernel(const uint8_t* w, uint8_t* out, int n, int k) {
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
  const int nn = nt * kTileN + q * 32 + t;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const int kk = kt * kTileK + j * 32 + c;
    out[(long long)kk * n + nn] = (uint8_t)((o[c >> 2] >> (8 * (c & 3))) & 0xFF);
  }
}

cudaError_t launch_debug_mx_codes(const uint8_t* w, uint8_t* out_kn, int64_t n, int64_t k,
                                  cudaStream_t stream) {
  const long long total = (n / kTileN) * (k / kTileK) * 512;
  debug_mx_codes_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(w, out_kn, (int)n,
                                                                           (int)k);
  return cudaGetLastError();
}

}  // namespace qg
