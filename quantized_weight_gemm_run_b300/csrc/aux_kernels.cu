// Memory-bound support kernels of the hot path: per-token FP8 activation
// quantization (W4A8 path), and the MoE permutation, SiLU gate and combine
// around the grouped GEMMs.
//
// The pages name the W4A8-MXFP4 path with FP8 activations (kinachrichten.com,
// "Kompilierzeiten und geraetespezifisches Tuning", MXFP4 paragraph) and MoE
// layers in which each token activates a subset of the experts (same article,
// "Warum quantisierte Kernel wichtig sind"); the arithmetic of each kernel is
// stated at the kernel.

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"

namespace qg {

// The checked build's word for the kernels of this file (they have no
// workspace); never written by the unchecked build.
__device__ int g_check_word = 0;

int checked_word_read_and_clear() {
  int w = 0;
  if (cudaMemcpyFromSymbol(&w, g_check_word, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  if (w && cudaMemcpyToSymbol(g_check_word, &zero, sizeof(int)) != cudaSuccess) return -1;
  return w;
}

// One index test that fails by construction (index 1 against an extent of
// 1); nothing is accessed through it.
__global__ void check_selftest_kernel(int* word, int extent) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    const int index = 1;
    if (qg_check(index < extent, word)) word[1] = index;   // never taken
  }
}

cudaError_t launch_check_selftest(int* word, cudaStream_t stream) {
  check_selftest_kernel<<<1, 32, 0, stream>>>(word, 1);
  return cudaGetLastError();
}

// Programmatic dependent launch for the auxiliary kernels.  Each waits for
// the previous grid on the stream to complete, memory included, before it
// touches memory (a no-op when launched without the attribute).  The
// activation quantization also lets the next grid begin launching at once,
// so the W4A8 GEMM's start-up (barriers, tensor memory, the first weight
// copy) overlaps it; it is launched with the attribute itself.  The MoE
// kernels neither overlap their own launch nor let the next grid start
// early: both measured 0.5-1.5 % slower per layer on B300.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream,
                              bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ----------------------------------------------------------- FP8 act quant
// One warp per row, four rows per CTA (spread over more SMs): s = max|x| / 448 (fp32, IEEE divide;
// 1 for an all-zero row), code = e4m3_rn_satfinite(x / s) with an IEEE fp32
// divide.  Lanes take 16-byte vectors (8 bf16) of the row in turn; the first
// kActVecs vectors of each lane stay in registers between the max and the
// quantization (a 2048-wide row in one pass), the rest of a longer row is read
// again.  Codes leave as 8-byte stores.
constexpr int kActVecs = 8;
constexpr int kActRowsPerCta = 4;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float absmax8(float amax, const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
  return amax;
}

__device__ __forceinline__ uint2 quant8(const uint4& v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = __nv_cvt_float_to_fp8(__fdiv_rn(bf16_lo(w[i]), s), __NV_SATFINITE,
                                              __NV_E4M3);
    const uint32_t hi = __nv_cvt_float_to_fp8(__fdiv_rn(bf16_hi(w[i]), s), __NV_SATFINITE,
                                              __NV_E4M3);
    o[i >> 1] |= (lo | (hi << 8)) << (16 * (i & 1));
  }
  return make_uint2(o[0], o[1]);
}

__global__ void __launch_bounds__(32 * kActRowsPerCta)
    act_quant_fp8_kernel(const uint4* __restrict__ x, int m, int kv, uint2* __restrict__ a8,
                         float* __restrict__ scale) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * kActRowsPerCta + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= m) return;
  const uint4* xr = x + (long long)row * kv;
  uint2* out = a8 + (long long)row * kv;
  uint4 v[kActVecs];
  float amax = 0.f;
#pragma unroll
  for (int c = 0; c < kActVecs; ++c) {
    const int i = lane + 32 * c;
    v[c] = i < kv ? __ldg(xr + i) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int c = 0; c < kActVecs; ++c) amax = absmax8(amax, v[c]);
  for (int i = lane + 32 * kActVecs; i < kv; i += 32) amax = absmax8(amax, __ldg(xr + i));
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
  if (lane == 0) scale[row] = s;
#pragma unroll
  for (int c = 0; c < kActVecs; ++c) {
    const int i = lane + 32 * c;
    if (i < kv) out[i] = quant8(v[c], s);
  }
  for (int i = lane + 32 * kActVecs; i < kv; i += 32) out[i] = quant8(__ldg(xr + i), s);
}

cudaError_t launch_act_quant_fp8(const uint16_t* x, int64_t m, int64_t k, uint8_t* a8,
                                 float* scale, cudaStream_t stream) {
  if (m == 0) return cudaSuccess;
  const unsigned ctas = (unsigned)((m + kActRowsPerCta - 1) / kActRowsPerCta);
  return launch_pdl(act_quant_fp8_kernel, dim3(ctas), dim3(32 * kActRowsPerCta), stream, true,
                    reinterpret_cast<const uint4*>(x), (int)m, (int)(k / 8),
                    reinterpret_cast<uint2*>(a8), scale);
}

// ----------------------------------------------------------- MoE permute
// Stable counting sort of the slots s = token*topk + j by expert id.  Ids
// outside [0, E) go to an extra bucket after the last expert, so perm is
// always a full permutation of the slots.
//
// The slots are cut into blocks of kSortBlock, one CTA (32 warps) each, and
// each block into 32 contiguous warp segments.  A slot's place is
//   (slots of lower experts) + (slots of its expert in earlier blocks)
//   + (... in earlier segments of its block) + (... earlier in its segment),
// the first three from per-block and per-warp histograms (order-free shared
// memory atomics), the last from a warp match over 32 consecutive slots.
// One block: a single kernel; more: a histogram kernel per block, then the
// placement kernel, which sums the blocks' histograms itself.
constexpr int kSortBlock = 2048;

__device__ __forceinline__ int sort_bucket(const int32_t* ids, int i, int E) {
  const int v = ids[i];
  return (v >= 0 && v < E) ? v : E;
}

// Per-block histograms: hist[blockIdx.x][e], e in [0, E].
__global__ void __launch_bounds__(1024) moe_count_kernel(const int32_t* __restrict__ ids,
                                                         int n_slots, int E,
                                                         int32_t* __restrict__ hist) {
  pdl_wait();
  constexpr int NB = kMaxPermuteExperts + 1;
  __shared__ int h[NB];
  const int B = E + 1;
  for (int x = threadIdx.x; x < B; x += blockDim.x) h[x] = 0;
  __syncthreads();
  const int lo = blockIdx.x * kSortBlock, hi = min(lo + kSortBlock, n_slots);
  for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) atomicAdd(&h[sort_bucket(ids, i, E)], 1);
  __syncthreads();
  for (int x = threadIdx.x; x < B; x += blockDim.x) hist[blockIdx.x * B + x] = h[x];
}

// Places the slots of block blockIdx.x.  hist: the per-block histograms of
// all nblocks blocks, or NULL when there is one block (counted here).
__global__ void __launch_bounds__(1024) moe_place_kernel(const int32_t* __restrict__ ids,
                                                         int n_slots, int E, int nblocks,
                                                         const int32_t* __restrict__ hist,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ perm,
                                                         int32_t* __restrict__ inv_perm) {
  pdl_wait();
  constexpr int NB = kMaxPermuteExperts + 1;
  __shared__ int cnt[32][NB];   // per-warp counts, then per-warp running bases
  __shared__ int start[NB];     // this block's first place per bucket
  __shared__ int tot[NB];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = E + 1;
  const int blo = blockIdx.x * kSortBlock, bhi = min(blo + kSortBlock, n_slots);
  for (int x = tid; x < 32 * NB; x += blockDim.x) (&cnt[0][0])[x] = 0;
  __syncthreads();
  const int seg = (bhi - blo + 31) / 32;
  const int lo = min(blo + warp * seg, bhi), hi = min(lo + seg, bhi);
  for (int i = lo + lane; i < hi; i += 32) atomicAdd(&cnt[warp][sort_bucket(ids, i, E)], 1);
  __syncthreads();
  // per bucket: exclusive scan over this block's warps; the block's own
  // total, and the slots of the bucket in earlier blocks
  for (int x = tid; x < B; x += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = cnt[w][x];
      cnt[w][x] = run;
      run += c;
    }
    int before = 0, all = run;
    if (hist) {
      all = 0;
      for (int b = 0; b < nblocks; ++b) {
        const int c = hist[b * B + x];
        if (b < (int)blockIdx.x) before += c;
        all += c;
      }
    }
    tot[x] = all;
    start[x] = before;
  }
  __syncthreads();
  if (warp == 0) {   // exclusive scan of the bucket totals: the expert offsets
    int carry = 0;
    for (int x0 = 0; x0 < B; x0 += 32) {
      const int x = x0 + lane;
      const int v = x < B ? tot[x] : 0;
      int incl = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += t;
      }
      if (x < B) {
        start[x] += carry + incl - v;
        if (blockIdx.x == 0 && x <= E) offsets[x] = carry + incl - v;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int i0 = lo; i0 < hi; i0 += 32) {
    const int i = i0 + lane;
    const int e = i < hi ? sort_bucket(ids, i, E) : -1;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int pos = start[e] + cnt[warp][e] + __popc(same & lt_mask);
      if (qg_check(pos >= 0 && pos < n_slots, &g_check_word)) {
        perm[pos] = i;
        inv_perm[i] = pos;
      }
    }
    __syncwarp();
    if (e >= 0 && (same & lt_mask) == 0) cnt[warp][e] += __popc(same);
    __syncwarp();
  }
}

// a_perm[r] = a[perm[r] / topk]: one warp per row, 16-byte vectors.
__global__ void gather_rows_kernel(const uint4* __restrict__ a, const int32_t* __restrict__ perm,
                                   uint4* __restrict__ a_perm, int rows, int topk, int vecs) {
  pdl_wait();
  const int warps = blockDim.x >> 5;
  const int r = blockIdx.x * warps + (threadIdx.x >> 5);
  if (r >= rows) return;
  if (!qg_check(perm[r] >= 0 && perm[r] < rows, &g_check_word)) return;
  const int src = perm[r] / topk;
  const uint4* s = a + (long long)src * vecs;
  uint4* d = a_perm + (long long)r * vecs;
  for (int v = threadIdx.x & 31; v < vecs; v += 32) d[v] = s[v];
}

cudaError_t launch_moe_permute(const int32_t* ids, int64_t t, int topk, int e, int32_t* offsets,
                               int32_t* perm, int32_t* inv_perm, const uint16_t* a,
                               uint16_t* a_perm, int64_t hidden, cudaStream_t stream) {
  const int n_slots = (int)(t * topk);
  const int nblocks = (n_slots + kSortBlock - 1) / kSortBlock;
  cudaError_t err;
  if (nblocks <= 1) {
    err = launch_pdl(moe_place_kernel, dim3(1), dim3(1024), stream, false, ids, n_slots, e, 1,
                     (const int32_t*)nullptr, offsets, perm, inv_perm);
  } else {
    // the per-block histograms (nblocks x (E + 1) ints, far smaller than the
    // gathered rows) live in a_perm, which the gather overwrites afterwards
    int32_t* hist = reinterpret_cast<int32_t*>(a_perm);
    err = launch_pdl(moe_count_kernel, dim3(nblocks), dim3(1024), stream, false, ids, n_slots, e,
                     hist);
    if (err != cudaSuccess) return err;
    err = launch_pdl(moe_place_kernel, dim3(nblocks), dim3(1024), stream, false, ids, n_slots, e,
                     nblocks, (const int32_t*)hist, offsets, perm, inv_perm);
  }
  if (err != cudaSuccess || n_slots == 0) return err;
  const int vecs = (int)(hidden * 2 / 16);
  return launch_pdl(gather_rows_kernel, dim3((n_slots + 7) / 8), dim3(256), stream, false,
      reinterpret_cast<const uint4*>(a), perm, reinterpret_cast<uint4*>(a_perm), n_slots, topk,
      vecs);
}

// ----------------------------------------------------------- SiLU gate
// h[r, i] = bf16(silu(g) * u), g = gu[r, i], u = gu[r, inter + i], fp32 math,
// silu(g) = g / (1 + exp(-g)).  Eight elements per thread.
__global__ void silu_mul_kernel(const uint16_t* __restrict__ gu, uint16_t* __restrict__ h,
                                long long rows, int inter) {
  pdl_wait();
  const int per_row = inter / 8;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * per_row) return;
  const long long r = idx / per_row;
  const int c = (int)(idx % per_row) * 8;
  const uint4 gv = *reinterpret_cast<const uint4*>(gu + r * 2 * inter + c);
  const uint4 uv = *reinterpret_cast<const uint4*>(gu + r * 2 * inter + inter + c);
  const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
  const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&uv);
  uint4 ov;
  __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&ov);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 g = __bfloat1622float2(g2[i]);
    const float2 u = __bfloat1622float2(u2[i]);
    o2[i] = __floats2bfloat162_rn(silu_mul_f32(g.x, u.x), silu_mul_f32(g.y, u.y));
  }
  *reinterpret_cast<uint4*>(h + r * inter + c) = ov;
}

cudaError_t launch_silu_mul(const uint16_t* gu, int64_t rows, int64_t inter, uint16_t* h,
                            cudaStream_t stream) {
  const long long total = rows * (inter / 8);
  if (total == 0) return cudaSuccess;
  return launch_pdl(silu_mul_kernel, dim3((unsigned)((total + 255) / 256)), dim3(256), stream,
                    false, gu, h, (long long)rows, (int)inter);
}

// ----------------------------------------------------------- combine
// y[t, :] = bf16(sum_j w[t, j] * y2[inv_perm[t*topk + j], :]), fp32, j in order.
__global__ void combine_kernel(const uint16_t* __restrict__ y2, const int32_t* __restrict__ inv_perm,
                               const float* __restrict__ w, uint16_t* __restrict__ y, int topk,
                               int hidden) {
  pdl_wait();
  const int t = blockIdx.x;
  const int c = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (c >= hidden) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  // eight slots at a time: every load of a batch is issued before the first
  // use, and the products are added in slot order
  for (int j0 = 0; j0 < topk; j0 += 8) {
    float wj[8];
    int r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j0 + j < topk) {
        wj[j] = w[(long long)t * topk + j0 + j];
        r[j] = inv_perm[(long long)t * topk + j0 + j];
      }
    }
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j0 + j < topk &&
          qg_check(r[j] >= 0 && r[j] < (int)gridDim.x * topk, &g_check_word))
        v[j] = *reinterpret_cast<const uint4*>(y2 + (long long)r[j] * hidden + c);
      else
        v[j] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j0 + j < topk) {
        const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&v[j]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(v2[i]);
          acc[2 * i] = fmaf(wj[j], f.x, acc[2 * i]);
          acc[2 * i + 1] = fmaf(wj[j], f.y, acc[2 * i + 1]);
        }
      }
    }
  }
  uint4 ov;
  __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&ov);
#pragma unroll
  for (int i = 0; i < 4; ++i) o2[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
  *reinterpret_cast<uint4*>(y + (long long)t * hidden + c) = ov;
}

cudaError_t launch_combine(const uint16_t* y2, const int32_t* inv_perm, const float* w, int64_t t,
                           int topk, int64_t hidden, uint16_t* y, cudaStream_t stream) {
  if (t == 0) return cudaSuccess;
  const int threads = 128;
  dim3 grid((unsigned)t, (unsigned)((hidden / 8 + threads - 1) / threads));
  return launch_pdl(combine_kernel, grid, dim3(threads), stream, false, y2, inv_perm, w, y, topk,
                    (int)hidden);
}

}  // namespace qg
