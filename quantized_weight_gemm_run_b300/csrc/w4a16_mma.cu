// Small-M W4A16 GEMM on register-fed tensor-core MMAs (mma.sync).
//
// The pages describe two pipelines for the same GEMM: a cp.async + MMA
// pipeline that can win at small batch and a TMA + UMMA pipeline for larger
// batch, and an M-range heuristic that picks between kernels per input size
// (kinachrichten.com, "Wie die Architektur funktioniert"; jetabc.cn,
// "Humming 的做法").  This is the small-batch one, for M <= 16 rows and the
// INT4 / UINT4 formats, on the same packed weight buffer as the tcgen05
// kernel.
//
// Shape.  Swap-AB again: D[n, m] = W^[n, :] . A[m, :], the 128 features of
// an n-tile as MMA rows (8 m16 blocks, two per warp) and the <= 16 tokens as
// two n8 blocks.  Dequantized weights go straight from registers into the A
// fragments: in the packed layout, lane t of a quad finds its (k, k+1) pairs
// at nibble positions t and t+4 of every 32-bit word, so a quad's four lanes
// read the same 16-byte vector (one broadcast) and each extracts its own pairs
// with one LOP3 against a magic exponent.  Activations come through ldmatrix
// from a padded shared-memory tile (conflict-free rows).
//
// Work split.  Grid = n-tiles x S K-slices, about five CTAs of 128 threads
// per SM; a CTA issues cp.async copies for its slice's k-tiles through a ring
// of kStages slots (the whole slice up front when it fits), weights before
// the wait on the previous grid, activations after it.  Partials: the CTA's
// m x 128 fp32 result rows are staged in shared memory and added into the
// n-tile's accumulator in L2 with one bulk reduction; the CTA then counts in
// with an acquire-release add, and the last of the S arrivals adds the bias,
// rounds, writes the output rows and re-zeroes the accumulator and counter.
// Nothing waits on another CTA, so no wait needs a time limit.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace qg {

namespace {

constexpr int kMmaThreads = 128;
constexpr int kStages = 3;
constexpr int kARowBytes = 272;                 // 128 k x 2 B, padded by 16 B
constexpr int kATileBytes = 16 * kARowBytes;    // 16 tokens

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

template <bool FP16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (FP16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// (magic + q) pair -> ((magic + q) - (magic + z)) * s, one rounding
template <bool FP16>
__device__ __forceinline__ uint32_t dq2(uint32_t word_shifted, uint32_t zero2, uint32_t scale2) {
  constexpr uint32_t magic = FP16 ? 0x64006400u : 0x43004300u;
  uint32_t x;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;"
      : "=r"(x)
      : "r"(word_shifted), "r"(0x000F000Fu), "r"(magic));
  if constexpr (FP16) {
    __half2 r = __hmul2(__hsub2(*reinterpret_cast<__half2*>(&x),
                                *reinterpret_cast<__half2*>(&zero2)),
                        *reinterpret_cast<__half2*>(&scale2));
    return *reinterpret_cast<uint32_t*>(&r);
  } else {
    __nv_bfloat162 r = __hmul2(__hsub2(*reinterpret_cast<__nv_bfloat162*>(&x),
                                       *reinterpret_cast<__nv_bfloat162*>(&zero2)),
                               *reinterpret_cast<__nv_bfloat162*>(&scale2));
    return *reinterpret_cast<uint32_t*>(&r);
  }
}

}  // namespace

// ONE_GROUP: the group size is >= 128, so one scale (and zero) per row
// serves the whole k-tile.
template <bool FP16, bool ONE_GROUP>
__global__ void __launch_bounds__(kMmaThreads) w4a16_mma_kernel(const W4A16MmaParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int nt = blockIdx.x / p.splits, sl = blockIdx.x - nt * p.splits;
  const int kt0 = (int)((long long)sl * p.kt / p.splits);
  const int kt1 = (int)((long long)(sl + 1) * p.kt / p.splits);
  const int nk = kt1 - kt0;
  const int slot_bytes = p.w_slot_bytes + kATileBytes;
  const uint8_t* wsrc = p.w + ((long long)nt * p.kt + kt0) * p.block_bytes;

  // stage s (k-tile kt0 + s): weight block into slot s % kStages, then its
  // activation tile (16 rows, zero-filled past m)
  auto issue_w = [&](int s) {
    if (s < nk) {
      uint8_t* dst = smem + (s % kStages) * slot_bytes;
      const uint8_t* src = wsrc + (long long)s * p.block_bytes;
      for (int c = tid; c < p.block_bytes / 16; c += kMmaThreads)
        cp_async16(dst + c * 16, src + c * 16, 16);
    }
  };
  auto issue_a = [&](int s) {
    if (s < nk) {
      uint8_t* dst = smem + (s % kStages) * slot_bytes + p.w_slot_bytes;
      const int kbase = (kt0 + s) * kTileK;
      for (int c = tid; c < 16 * 16; c += kMmaThreads) {   // 16 rows x 16 chunks of 16 B
        const int r = c >> 4, ch = c & 15;
        const bool live = r < p.m;
        const uint16_t* src = p.a + (long long)(live ? r : 0) * p.k + kbase + ch * 8;
        cp_async16(dst + r * kARowBytes + ch * 16, src, live ? 16 : 0);
      }
    }
  };

  // weights are read-only layer data: stream them before the wait
#pragma unroll 1
  for (int s = 0; s < kStages - 1; ++s) issue_w(s);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#pragma unroll 1
  for (int s = 0; s < kStages - 1; ++s) {
    issue_a(s);
    cp_async_commit();
  }

  float acc[2][2][4];
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[b][c][i] = 0.f;

  constexpr uint32_t magic16 = FP16 ? 0x6400u : 0x4300u;
#pragma unroll 1
  for (int s = 0; s < nk; ++s) {
    issue_w(s + kStages - 1);
    issue_a(s + kStages - 1);
    cp_async_commit();
    cp_async_wait<kStages - 1>();   // stage s has landed
    __syncthreads();
    const uint8_t* slot = smem + (s % kStages) * slot_bytes;
    const uint4* wv = reinterpret_cast<const uint4*>(slot);
    const uint16_t* sv = reinterpret_cast<const uint16_t*>(slot + p.s_off);
    const uint8_t* zv = slot + p.z_off;
    const uint8_t* at = slot + p.w_slot_bytes;
    // per-row scale and zero pairs of rows (b, g) and (b, g + 8), group sg
    auto row_consts = [&](int sg, uint32_t (&sc)[2][2], uint32_t (&zc)[2][2]) {
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = warp * 32 + b * 16 + g + 8 * e;
          sc[b][e] = (uint32_t)sv[sg * kTileN + r] * 0x00010001u;
          zc[b][e] = (magic16 + (p.has_zp ? (uint32_t)zv[sg * kTileN + r] : 8u)) * 0x00010001u;
        }
    };
    uint32_t sc[2][2], zc[2][2];
    if constexpr (ONE_GROUP) row_consts(0, sc, zc);
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // 32-k chunk
      // B fragments of the chunk's two k16 steps, tokens 0-7 and 8-15
      uint32_t bf[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int mi = lane >> 3;   // matrix: (tokens 8 (mi >> 1) .., k + 8 (mi & 1))
        const int tok = (mi >> 1) * 8 + (lane & 7);
        ldmatrix_x4(bf[h], at + tok * kARowBytes + (j * 32 + h * 16 + (mi & 1) * 8) * 2);
      }
      if constexpr (!ONE_GROUP) row_consts(j >> p.sg_shift, sc, zc);
#pragma unroll
      for (int b = 0; b < 2; ++b) {   // m16 block: rows 32 warp + 16 b + {g, g + 8}
        const uint4 v0 = wv[(warp * 4 + j) * 32 + b * 16 + g];
        const uint4 v1 = wv[(warp * 4 + j) * 32 + b * 16 + g + 8];
        const uint32_t s0 = sc[b][0], s1 = sc[b][1], z0 = zc[b][0], z1 = zc[b][1];
        const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
        const uint32_t w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {   // k16 step: words 2h (k 0-7) and 2h+1 (k 8-15)
          uint32_t af[4];
          af[0] = dq2<FP16>(w0[2 * h] >> (4 * t), z0, s0);
          af[1] = dq2<FP16>(w1[2 * h] >> (4 * t), z1, s1);
          af[2] = dq2<FP16>(w0[2 * h + 1] >> (4 * t), z0, s0);
          af[3] = dq2<FP16>(w1[2 * h + 1] >> (4 * t), z1, s1);
          mma16816<FP16>(acc[b][0], af, bf[h][0], bf[h][1]);
          mma16816<FP16>(acc[b][1], af, bf[h][2], bf[h][3]);
        }
      }
    }
    __syncthreads();   // the slot is rewritten by the next issue
  }
  cp_async_wait<0>();

  // the CTA's partial as [token][128 features] fp32 in slot 0: the m live
  // token rows are contiguous, so only they are reduced, read and re-zeroed
  float* cs = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int f = warp * 32 + b * 16 + g, tk = c * 8 + 2 * t;
      cs[tk * kTileN + f] = acc[b][c][0];
      cs[(tk + 1) * kTileN + f] = acc[b][c][1];
      cs[tk * kTileN + f + 8] = acc[b][c][2];
      cs[(tk + 1) * kTileN + f + 8] = acc[b][c][3];
    }
  fence_proxy_async_smem();   // every writer, before the bulk reduction reads the tile
  __syncthreads();

  __shared__ int last;
  const float* sum = cs;   // where the finished fp32 rows are read from
  if (p.splits > 1) {
    float* tile = p.acc + (long long)nt * (kTileN * 16);
    if (tid == 0) {
      bulk_reduce_add_f32(tile, cs, p.m * kTileN * 4);
      bulk_commit_group();
      bulk_wait_group_all();
      asm volatile("fence.proxy.async.global;" ::: "memory");
      int old;
      asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                   : "=r"(old)
                   : "l"(p.counters + nt)
                   : "memory");
      last = (old == p.splits - 1);
    }
    __syncthreads();
    if (!last) return;
    sum = tile;
  }
  // finish: thread f owns feature f of the n-tile
  const int f = tid;
  const int n = nt * kTileN + f;
  float bias = 0.f;
  if (p.bias) {
    const uint16_t bb = p.bias[n];
    bias = FP16 ? __half2float(*reinterpret_cast<const __half*>(&bb))
                : __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(&bb));
  }
  // every live row's sum is loaded before the first output store (the stores
  // could alias the loads as far as the compiler knows, which would serialize
  // them one L2 round trip each)
  float v[16];
#pragma unroll
  for (int r = 0; r < 16; ++r)
    v[r] = r < p.m ? (p.splits > 1 ? __ldcg(sum + r * kTileN + f) : sum[r * kTileN + f]) : 0.f;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    if (r < p.m) {
      uint16_t o;
      if constexpr (FP16) {
        const __half h = __float2half_rn(v[r] + bias);
        o = *reinterpret_cast<const uint16_t*>(&h);
      } else {
        const __nv_bfloat16 h = __float2bfloat16_rn(v[r] + bias);
        o = *reinterpret_cast<const uint16_t*>(&h);
      }
      p.c[(long long)r * p.n + n] = o;
    }
  }
  if (p.splits > 1) {   // leave the accumulator rows and the count at zero
    float* z = p.acc + (long long)nt * (kTileN * 16) + f;
#pragma unroll
    for (int r = 0; r < 16; ++r)
      if (r < p.m) z[r * kTileN] = 0.f;
    if (tid == 0) p.counters[nt] = 0;
  }
}

int mma_smem_bytes(int block_bytes) {
  return kStages * (((block_bytes + 15) & ~15) + kATileBytes);
}

cudaError_t launch_w4a16_mma(const W4A16MmaParams& p, bool fp16, cudaStream_t stream) {
  const int smem = mma_smem_bytes(p.block_bytes);
  const bool one = p.sg_shift == 2;   // group >= 128
  auto kern = fp16 ? (one ? w4a16_mma_kernel<true, true> : w4a16_mma_kernel<true, false>)
                   : (one ? w4a16_mma_kernel<false, true> : w4a16_mma_kernel<false, false>);
  static int attr_set[4] = {0, 0, 0, 0};
  int& done = attr_set[(fp16 ? 2 : 0) + (one ? 1 : 0)];
  if (smem > done) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    done = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.nt * p.splits));
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace qg
