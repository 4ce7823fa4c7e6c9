// W4A4: NVFP4 weights against NVFP4 activations on the block-scaled FP4
// tensor cores (tcgen05.mma kind::mxf4nvf4).  The pages list W4A4 among the
// common configurations and name NVFP4 (e2m1 codes with an e4m3 scale per 16
// elements and an fp32 tensor scale) as a format whose number format and
// scaling differ from INT4's (kinachrichten.com, "Warum quantisierte Kernel
// wichtig sind").
//
// Two kernels:
//   act_quant_nvfp4_kernel  bf16 activations -> e2m1 codes and e4m3 block
//                           scales per 16 k of each token, against the
//                           caller's fp32 tensor scale (every decision in
//                           fp32: d = 6 a_ts, t = amax / d, s = e4m3(t),
//                           q = x / (s a_ts), code = e2m1(q))
//   w4a4_kernel<BT>         persistent, one CTA per SM over the work items
//                           (a BT-token, 128-feature tile, or one of its S
//                           contiguous K slices): both operands stay packed
//                           (two codes a byte) from HBM to the tensor core,
//                           the block scales go to tensor memory, and the
//                           epilogue multiplies the fp32 sums by the two
//                           tensor scales; two accumulators let an item's
//                           epilogue run under the next item's MMAs.  With
//                           S > 1 (few tiles: small M) each slice's epilogue
//                           writes its fp32 partial to the workspace and the
//                           last slice of a tile to count in sums the S
//                           partials in slice order (the bits do not depend
//                           on which slice finishes last) before the scales,
//                           bias and rounding; its counters are cleared by
//                           the quantization kernel ahead of it.
//
// Roles of the 12 warps: 0 TMA producer, 1 MMA issuer, 2 tensor-memory
// allocation, 4-7 block scales into tensor memory, 8-11 the epilogue (warps
// w and w + 4 own tensor-memory lanes 32 (w - 4) ... + 31).
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace qg {
namespace {

constexpr int kStages = 6;      // pipeline depth (256 k a stage)
constexpr int kThreads = 384;

template <int BT>
struct Lay {
  static constexpr int kA = 128 * 128;   // weight codes: 128 features x 128 bytes (256 k)
  static constexpr int kB = BT * 128;    // activation codes
  static constexpr int kSA = 128 * 16;   // weight block scales: 128 x 16 bytes
  static constexpr int kSB = BT * 16;    // activation block scales
  static constexpr int kOffB = kA;
  static constexpr int kOffSA = kA + kB;
  static constexpr int kOffSB = kA + kB + kSA;
  static constexpr int kBytes = kA + kB + kSA + kSB;           // TMA bytes a stage
  static constexpr int kStage = (kBytes + 1023) / 1024 * 1024;  // 1 KB aligned (swizzle atoms)
  static constexpr int kBar = kStages * kStage;
  static constexpr int kSmem = 1024 + kBar + 256;   // alignment slack, ring, barriers
  // tensor memory: two accumulators in columns [0, 2 BT), then per stage and
  // K=64 step a group of four columns of weight scales and a group of four
  // of activation scales.  A group holds the 32-bit scale words (byte i: the
  // scale of the step's 16-k block i) of 128 rows, row r in column r / 32 at
  // lane r mod 32 of every 32-lane quadrant (each quadrant of the tensor
  // core reads its own copy); a group starts on a multiple of four columns.
  static constexpr int kColSA = 2 * BT;
  static constexpr int kColSB = 2 * BT + 16 * kStages;
  static constexpr int kUsed = 2 * BT + 32 * kStages;
  static constexpr int kCols = kUsed <= 128 ? 128 : kUsed <= 256 ? 256 : 512;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         const W4A4Params& p, int site) {
  return mbar_wait(bar, parity, abort_flag, p.status, p.wait_limit_ns, kStatusTimeout | site);
}

__device__ __forceinline__ int atomic_add_acq_rel(int* addr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(addr), "r"(v)
               : "memory");
  return old;
}

// Bounded wait that ignores the abort flag: at exit, lets the copies and
// MMAs already issued finish before their shared or tensor memory goes away.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer();
  while (globaltimer() - t0 < limit_ns)
    if (mbar_try_wait(bar, parity)) return;
}

template <int BT>
__global__ void __launch_bounds__(kThreads, 1)
    w4a4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_a,
                const __grid_constant__ CUtensorMap tm_ws,
                const __grid_constant__ CUtensorMap tm_as, const W4A4Params p) {
  using L = Lay<BT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + kStages;
  uint64_t* sf_full = empty + kStages;
  uint64_t* acc_full = sf_full + kStages;   // two accumulator buffers
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int S = p.splits;
  const int items = p.mt * p.nt * S;
  // item -> tile t = item / S, its K slice [kt_lo, kt_hi) of 256-k stages
  auto kt_lo = [&](int item) { return (item % S) * p.kt / S; };
  auto kt_hi = [&](int item) { return (item % S + 1) * p.kt / S; };
  const uint64_t drain_ns = p.wait_limit_ns + 1000000000ull;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, L::kCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_ws);
    prefetch_tmap(&tm_as);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Persistent: CTA b takes items b, b + grid, ...; item it is slice it % S
  // of tile t = it / S, and tile t is (token tile t / nt, feature tile
  // t % nt).  The stage ring runs on across items (stage use g = the CTA's
  // running count of 256-k stages).
  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      // The first item's first stages of weights (read-only layer data) go
      // out before the wait on the quantization kernel ahead on the stream
      // (programmatic dependent launch); the activations after it.
      const int it0 = blockIdx.x;   // < items: the grid is at most the items
      const int pre = min(kStages, kt_hi(it0) - kt_lo(it0));
      {
        const int n0 = ((it0 / S) % p.nt) * 128;
        for (int u = 0; u < pre; ++u) {
          uint8_t* st = smem + u * L::kStage;
          mbar_arrive_expect_tx(&full[u], L::kBytes);
          tma_load_2d(st, &tm_w, &full[u], (kt_lo(it0) + u) * 128, n0);
          tma_load_2d(st + L::kOffSA, &tm_ws, &full[u], (kt_lo(it0) + u) * 16, n0);
        }
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int g = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < items; it += gridDim.x) {
        const int t = it / S;
        const int n0 = (t % p.nt) * 128, m0 = (t / p.nt) * BT;
        for (int kt = kt_lo(it); kt < kt_hi(it); ++kt, ++g) {
          const int s = g % kStages;
          if (g >= kStages &&
              !wait_bar(&empty[s], ((g / kStages) - 1) & 1, abort_flag, p, kSiteW4A4Slot)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * L::kStage;
          if (g >= pre) {   // else its weights went out before the wait
            mbar_arrive_expect_tx(&full[s], L::kBytes);
            tma_load_2d(st, &tm_w, &full[s], kt * 128, n0);
            tma_load_2d(st + L::kOffSA, &tm_ws, &full[s], kt * 16, n0);
          }
          tma_load_2d(st + L::kOffB, &tm_a, &full[s], kt * 128, m0);
          tma_load_2d(st + L::kOffSB, &tm_as, &full[s], kt * 16, m0);
        }
      }
      // let the copies already issued land before the CTA may exit
      for (int u = g > kStages ? g - kStages : 0; u < g; ++u)
        drain_bar(&full[u % kStages], (u / kStages) & 1, drain_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_mxf4nvf4_e2m1(BT);
      int g = 0, i = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < items; it += gridDim.x, ++i) {
        const int b = i & 1;
        if (!wait_bar(&acc_empty[b], ((i >> 1) & 1) ^ 1, abort_flag, p, kSiteW4A4Acc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + b * BT;
        const int k_first = kt_lo(it);
        for (int kt = k_first; kt < kt_hi(it); ++kt, ++g) {
          const int s = g % kStages;
          const uint32_t ph = (g / kStages) & 1;
          if (!wait_bar(&full[s], ph, abort_flag, p, kSiteW4A4Full) ||
              !wait_bar(&sf_full[s], ph, abort_flag, p, kSiteW4A4Scales)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * L::kStage), b0 = a0 + L::kOffB;
#pragma unroll
          for (int j = 0; j < 4; ++j)   // four K=64 steps of 32 bytes through each 128-byte row
            mma_ss_mxf4nvf4(d_tmem, smem_desc_sw128(a0 + 32 * j), smem_desc_sw128(b0 + 32 * j),
                            idesc, tmem + L::kColSA + 16 * s + 4 * j,
                            tmem + L::kColSB + 16 * s + 4 * j,
                            (kt > k_first || j > 0) ? 1u : 0u);
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&acc_full[b]);
      }
      mma_commit(drain);   // arrives once every MMA issued above has finished
      drain_bar(drain, 0, drain_ns);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------ block scales into tensor memory
    const uint32_t lane_addr = (uint32_t)((warp - 4) * 32) << 16;
    bool ok = true;
    int g = 0;
    for (int it = blockIdx.x; ok && it < items; it += gridDim.x) {
      for (int kt = kt_lo(it); kt < kt_hi(it); ++kt, ++g) {
        const int s = g % kStages;
        if (lane == 0) ok = wait_bar(&full[s], (g / kStages) & 1, abort_flag, p, kSiteW4A4Full);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        const uint8_t* st = smem + s * L::kStage;
        // this quadrant's copy of the stage's four scale groups: column
        // 4j + c holds word j (the scales of step j's four 16-k blocks) of
        // row 32 c + lane; activation rows past the tile hold zero
        uint32_t va[16], vb[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int row = 32 * c + lane;
          const uint4 a4 = *reinterpret_cast<const uint4*>(st + L::kOffSA + row * 16);
          uint4 b4 = make_uint4(0u, 0u, 0u, 0u);
          if (row < BT) b4 = *reinterpret_cast<const uint4*>(st + L::kOffSB + row * 16);
          va[c] = a4.x, va[4 + c] = a4.y, va[8 + c] = a4.z, va[12 + c] = a4.w;
          vb[c] = b4.x, vb[4 + c] = b4.y, vb[8 + c] = b4.z, vb[12 + c] = b4.w;
        }
        tmem_st16(tmem + lane_addr + L::kColSA + 16 * s, va);
        tmem_st16(tmem + lane_addr + L::kColSB + 16 * s, vb);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_full[s]);
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------ epilogue
    const int q = warp - 8;
    const int col = q * 32 + lane;   // feature within the tile
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    // the counters and the output: after the quantization kernel is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float sc = __fmul_rn(*p.a_ts, *p.w_ts);
    int i = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x, ++i) {
      const int t = it / S;
      const int b = i & 1;
      bool ok = true;
      if (lane == 0) ok = wait_bar(&acc_full[b], (i >> 1) & 1, abort_flag, p, kSiteW4A4Acc);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int n = (t % p.nt) * 128 + col, m0 = (t / p.nt) * BT;
      const int live = min(BT, p.m - m0);   // tokens of this tile
      float bias = 0.f;
      if (p.bias && qg_check(n < p.n, p.status))
        bias = __bfloat162float(__ushort_as_bfloat16(p.bias[n]));
      // this slice's partial (item it = t * S + slice), [token][128 features]
      float* slot = p.part + (size_t)it * (BT * 128) + col;
#pragma unroll 1
      for (int c0 = 0; c0 < BT; c0 += 16) {
        uint32_t v[16];
        tmem_ld16_wait(tmem + lane_addr + b * BT + c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tl = c0 + j;
          if (tl < live && qg_check(n < p.n, p.status)) {
            if (S == 1) {
              const float o = fmaf(__uint_as_float(v[j]), sc, bias);
              p.c[(long long)(m0 + tl) * p.n + n] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
            } else if (qg_check((long long)it * BT + tl < p.part_rows, p.status)) {
              __stcg(slot + tl * 128, __uint_as_float(v[j]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      if (S > 1) {
        // count this quadrant's slice in; the last of the S sums them
        __threadfence();
        __syncwarp();
        int before = 0;
        if (lane == 0 && qg_check(t * 4 + q < p.cnt_words, p.status))
          before = atomic_add_acq_rel(p.cnt + t * 4 + q, 1);
        __syncwarp();
        before = __shfl_sync(0xFFFFFFFFu, before, 0);
        if (before == S - 1) {
          __threadfence();
          // 16 rows at a time, the S slices added in slice order; two slices'
          // loads (32 per lane) are in flight at once
          const float* base = p.part + (size_t)t * S * (BT * 128) + col;
          constexpr size_t kSl = (size_t)BT * 128;   // floats between slices
          // checked build: the tile's last partial row lies inside the region
          if (!qg_check(((long long)t * S + S) * BT <= p.part_rows, p.status)) continue;
#pragma unroll 1
          for (int c0 = 0; c0 < live; c0 += 16) {
            const float* b0 = base + (size_t)c0 * 128;
            float acc[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = c0 + j < live ? __ldcg(b0 + j * 128) : 0.f;
            int sl = 1;
#pragma unroll 1
            for (; sl + 1 < S; sl += 2) {
              float v1[16], v2[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                v1[j] = c0 + j < live ? __ldcg(b0 + sl * kSl + j * 128) : 0.f;
                v2[j] = c0 + j < live ? __ldcg(b0 + (sl + 1) * kSl + j * 128) : 0.f;
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) acc[j] = (acc[j] + v1[j]) + v2[j];
            }
            if (sl < S) {
              float v1[16];
#pragma unroll
              for (int j = 0; j < 16; ++j)
                v1[j] = c0 + j < live ? __ldcg(b0 + sl * kSl + j * 128) : 0.f;
#pragma unroll
              for (int j = 0; j < 16; ++j) acc[j] += v1[j];
            }
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c0 + j < live && qg_check(n < p.n, p.status)) {
                const float o = fmaf(acc[j], sc, bias);
                p.c[(long long)(m0 + c0 + j) * p.n + n] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(o));
              }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, L::kCols);
}

// One thread per 16-k block of a token: two 16-byte loads, the block maximum,
// the e4m3 scale, sixteen fp32 divides and e2m1 conversions, one 8-byte code
// store and one scale byte.  Threads 0 .. n_zero - 1 also clear the GEMM's
// K-split counters (the GEMM that follows on the stream counts from zero,
// whatever another plan left in the workspace).
__global__ void __launch_bounds__(256)
    act_quant_nvfp4_kernel(const uint16_t* __restrict__ x, int64_t m, int64_t k,
                           const float* __restrict__ a_ts, uint8_t* __restrict__ codes,
                           uint8_t* __restrict__ sb, int* __restrict__ zero_words,
                           int n_zero) {
  // programmatic dependent launch: the previous grid's memory first; the
  // GEMM that follows may start its set-up and weight copies at once
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t nb = k >> 4;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n_zero) zero_words[i] = 0;
  if (i >= m * nb) return;
  const int64_t row = i / nb, b = i - row * nb;
  const uint4* src = reinterpret_cast<const uint4*>(x + row * k + b * 16);
  const uint4 u0 = src[0], u1 = src[1];
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  float f[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {   // bf16 -> fp32 is exact: the bits move up
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
  const float ts = *a_ts;
  const float t = __fdiv_rn(amax, __fmul_rn(6.0f, ts));
  const __nv_fp8_storage_t sbyte = __nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
  const float s = __half2float(__half(__nv_cvt_fp8_to_halfraw(sbyte, __NV_E4M3)));
  const float den = __fmul_rn(s, ts);
  uint32_t lo = 0, hi = 0;
  if (den > 0.f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 qq = make_float2(__fdiv_rn(f[2 * j], den), __fdiv_rn(f[2 * j + 1], den));
      const uint32_t byte = __nv_cvt_float2_to_fp4x2(qq, __NV_E2M1, cudaRoundNearest);
      if (j < 4) lo |= byte << (8 * j);
      else hi |= byte << (8 * (j - 4));
    }
  }
  *reinterpret_cast<uint2*>(codes + row * (k >> 1) + b * 8) = make_uint2(lo, hi);
  sb[row * nb + b] = sbyte;
}

template <int BT>
cudaError_t launch_bt(const CUtensorMap& tm_w, const CUtensorMap& tm_a, const CUtensorMap& tm_ws,
                      const CUtensorMap& tm_as, const W4A4Params& p, cudaStream_t stream) {
  using L = Lay<BT>;
  static bool attr_set = false;   // the shared-memory opt-in, once per process
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(w4a4_kernel<BT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int items = p.mt * p.nt * p.splits;
  const int sms = device_sm_count();
  const int grid = sms > 0 && items > sms ? sms : items;   // one persistent CTA per SM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, w4a4_kernel<BT>, tm_w, tm_a, tm_ws, tm_as, p);
}

}  // namespace

int w4a4_smem_bytes(int block_tok) {
  switch (block_tok) {
    case 16: return Lay<16>::kSmem;
    case 32: return Lay<32>::kSmem;
    case 64: return Lay<64>::kSmem;
    case 128: return Lay<128>::kSmem;
    default: return 0;
  }
}

cudaError_t launch_w4a4(const CUtensorMap& tm_w, const CUtensorMap& tm_a, const CUtensorMap& tm_ws,
                        const CUtensorMap& tm_as, const W4A4Params& p, int block_tok,
                        cudaStream_t stream) {
  switch (block_tok) {
    case 16: return launch_bt<16>(tm_w, tm_a, tm_ws, tm_as, p, stream);
    case 32: return launch_bt<32>(tm_w, tm_a, tm_ws, tm_as, p, stream);
    case 64: return launch_bt<64>(tm_w, tm_a, tm_ws, tm_as, p, stream);
    case 128: return launch_bt<128>(tm_w, tm_a, tm_ws, tm_as, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_act_quant_nvfp4(const uint16_t* x, int64_t m, int64_t k, const float* a_ts,
                                   uint8_t* codes, uint8_t* sb, cudaStream_t stream,
                                   int* zero_words, int n_zero) {
  const int64_t blocks = std::max<int64_t>(m * (k >> 4), n_zero);
  if (blocks == 0) return cudaSuccess;
  const int64_t grid = (blocks + 255) / 256;
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, act_quant_nvfp4_kernel, x, m, k, a_ts, codes, sb, zero_words,
                            n_zero);
}

}  // namespace qg
