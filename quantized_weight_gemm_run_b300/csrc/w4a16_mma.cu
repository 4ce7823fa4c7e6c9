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
// Shape.  Swap-AB: D[n, m] = W^[n, :] . A[m, :], the 128 features of an
// n-tile as MMA rows (8 m16 blocks, two per warp) and the tokens as one n8
// block (M <= 8) or two.  Dequantized weights go straight from registers into
// the A fragments: in the packed layout, lane t of a quad finds its (k, k+1)
// pairs at nibble positions t and t+4 of every 32-bit word, so a quad's four
// lanes read the same 16-byte vector (one broadcast) and each extracts its
// own pairs with one LOP3 against a magic exponent.  Activations come through
// ldmatrix from a padded shared-memory tile (conflict-free rows).
//
// Work split.  One thread-block cluster of S CTAs per n-tile; CTA r of the
// cluster takes the r-th of S contiguous K slices.  Data movement is the TMA
// engine completing on mbarriers: the CTA's first weight blocks go out at
// entry as bulk copies, before the wait on the previous grid (packed weights
// are read-only layer data), together with an L2 prefetch of its activation
// rows; after the wait one 3-D tensor copy lands the slice's activations
// (rows past M and k past K read as zeros) in the 128-byte-swizzled layout
// that ldmatrix reads without bank conflicts.  When the ring is shorter than
// the slice, each warp releases a slot on an mbarrier and warp s % 4 refills
// slot s once all four have.  Each warp keeps two accumulator sets (even and
// odd k16 steps) so that its MMA chains are half as long.
//
// Reduction.  Each CTA pushes feature slice r of its [tokens][128] fp32
// partial into cluster peer r's receive buffer (st.async, counted on the
// peer's mbarrier, armed before a cluster barrier at entry); CTA r sums the S
// slices it receives in cluster-rank order (fixed order: the bits repeat run
// to run and do not depend on M), adds the bias, rounds and stores.  No
// workspace accumulators, no global atomics, no barrier at the end.
//
// Waits.  Every mbarrier wait is bounded (the process-wide wait limit); a CTA
// that gives up records a timeout in the workspace status word, skips the
// rest of its work but still sends its (meaningless) slices so that every
// peer completes, and waits (with a fixed bound) for its own copies and
// incoming slices to land before it exits.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace qg {

namespace {

// four warps: warp w takes rows 32 w .. 32 w + 31 of the n-tile
constexpr int kMmaWarps = 4;
constexpr int kMmaThreads = 32 * kMmaWarps;
constexpr unsigned long long kDrainLimitNs = 100000000ull;

// Not volatile: the compiler may interleave these with the independent
// dequant chains (a warp issues in order, so the schedule is what hides the
// latencies); the memory clobber keeps them after the barrier waits that
// publish the activation tile.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr)
      : "memory");
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t addr) {
  asm("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
      : "=r"(r[0]), "=r"(r[1])
      : "r"(addr)
      : "memory");
}

template <bool FP16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  // register-only: free for the compiler to schedule
  if constexpr (FP16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// The dequant of a (k, k+1) pair, in three stages:
// nibbles at bits 0-3 and 16-19 -> (magic + q) pair (exact), minus the
// (magic + z) pair (exact: q - z), times the scale pair (the one rounding).
template <bool FP16>
__device__ __forceinline__ uint32_t nib_pairs(uint32_t word_shifted) {
  constexpr uint32_t magic = FP16 ? 0x64006400u : 0x43004300u;
  uint32_t x;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;"
      : "=r"(x)
      : "r"(word_shifted), "r"(0x000F000Fu), "r"(magic));
  return x;
}

template <bool FP16>
__device__ __forceinline__ uint32_t sub2(uint32_t x, uint32_t zero2) {
  if constexpr (FP16) {
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<__half2*>(&zero2));
    return *reinterpret_cast<uint32_t*>(&r);
  } else {
    __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&x),
                               *reinterpret_cast<__nv_bfloat162*>(&zero2));
    return *reinterpret_cast<uint32_t*>(&r);
  }
}

template <bool FP16>
__device__ __forceinline__ uint32_t mul2(uint32_t x, uint32_t scale2) {
  if constexpr (FP16) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<__half2*>(&scale2));
    return *reinterpret_cast<uint32_t*>(&r);
  } else {
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&x),
                               *reinterpret_cast<__nv_bfloat162*>(&scale2));
    return *reinterpret_cast<uint32_t*>(&r);
  }
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// D = A . B (fresh: C = 0), m16n8k32, e4m3 operands, fp32 result.
__device__ __forceinline__ void mma16832_e4m3(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// Four e2m1 codes (bits 0-15 of c16, k in nibble order from the low end) ->
// four e4m3 bytes in k order, exactly (every e2m1 value is an e4m3 value):
// a byte-table lookup of the 3-bit magnitude's e4m3 byte, a sign-replicating
// byte permute that turns each code's sign bit into bit 6 of its byte, and
// one LOP3 that moves it to bit 7.  Only the selector's low 16 bits count.
__device__ __forceinline__ uint32_t e2m1x4_e4m3(uint32_t c16) {
  constexpr uint32_t kLo = 0x3C383000u;   // e4m3 of 0, 0.5, 1, 1.5
  constexpr uint32_t kHi = 0x4C484440u;   // e4m3 of 2, 3, 4, 6
  uint32_t mag, sgn, out;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(mag) : "r"(kLo), "r"(kHi), "r"(c16 & 0x7777u));
  asm("prmt.b32 %0, %1, %1, %2;" : "=r"(sgn) : "r"(0x80808080u), "r"(c16));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(out) : "r"(sgn << 1), "r"(0x80808080u), "r"(mag));
  return out;
}

// An e8m0 block scale 2^(b - 127) as fp32 (b = 0: the subnormal 2^-127).
__device__ __forceinline__ float e8m0_f32(uint32_t b) {
  return __uint_as_float(b ? b << 23 : 0x00400000u);
}

// L2 prefetch of a global range (16-byte aligned start, size a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

}  // namespace

// Shared-memory geometry of one CTA: the activation tile (one TMA box:
// 2 nk_max chunks of 64 k x rows x 128 bytes, 128-byte swizzled, at offset 0
// for the swizzle's 1 KB alignment), the weight ring, the receive buffer of
// the reduction ([S][rows][128 / S] fp32), then barriers and counters.
__host__ __device__ inline int mma_act_bytes(int nk_max, int rows, int elem_bytes) {
  return nk_max * rows * kTileK * elem_bytes;
}

int mma_smem_bytes(int block_bytes, int ring, int nk_max, int rows, int elem_bytes,
                   bool quant) {
  // quant: the bf16 box, then the e4m3 tile quantized from it, the partial
  // row maxima of the S slices and the rows' scales
  const int act = quant ? mma_act_bytes(nk_max, rows, 2) + mma_act_bytes(nk_max, rows, 1)
                        : mma_act_bytes(nk_max, rows, elem_bytes);
  return 1024 /* alignment slack */ + act + ring * block_bytes + rows * kTileN * 4 +
         (quant ? (16 + 1) * rows * 4 : 0) + 8 * (2 * ring + 3) + 16;
}

// NB: n8 token blocks (1: M <= 8, 2: M <= 16).  ONE_GROUP: the group size is
// >= 128, so one scale (and zero) per row serves the whole k-tile.  MX: W4A8
// (MXFP4 weights against e4m3 activations with per-row fp32 scales, bf16
// output): the codes become e4m3 bytes exactly, each 32-k block is one
// m16n8k32 e4m3 MMA into a fresh fp32 partial, and the partial is added with
// the block's scale 2^E (an exact power-of-two multiply) into the accumulator;
// the per-row activation scale multiplies the finished sum.
// QA (with MX): the activations arrive as bf16 and are quantized here, per
// row to e4m3 with the fp32 scale max|x| / 448, exactly as the standalone
// quantizer does: each CTA takes the maximum over its K slice, the cluster's S
// slices exchange their maxima through distributed shared memory (the max is
// exact, so every CTA derives the same scale), and each CTA quantizes its own
// slice into the e4m3 tile the MMAs read.
// F16S: bf16 activations with fp16 scales; each scale is split once per row
// into two bf16 terms (split_f16_scale) and w^ = fma(d, s_hi, d s_lo) rounds
// (q - z) s once, the dequantized values of the tcgen05 kernel's FMT 5.
// NV: NVFP4 weights (e2m1 codes in nibble order, one 16-bit block scale per
// 16 k, an fp32 tensor scale) against 16-bit activations: a lane's two codes
// of k 2t, 2t + 1 (and 2t + 8, 2t + 9) are byte t of words 2h and 2h + 1 of
// its row's vector; one prmt gathers both bytes, e2m1x4_pairs gives the exact
// 16-bit pairs, one multiply by the block scale rounds nothing (the products
// are exact), and the tensor scale multiplies the finished sum, as in the
// tcgen05 kernel.
template <bool FP16, int NB, bool ONE_GROUP, bool MX, bool QA = false, bool F16S = false,
          bool NV = false>
__global__ void __launch_bounds__(kMmaThreads, 4)
    w4a16_mma_kernel(const __grid_constant__ CUtensorMap tmap_a, const W4A16MmaParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzled activation box needs a 1 KB aligned start
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr int ROWS = 8 * NB;
  static_assert(!QA || MX, "activation quantization serves the W4A8 path");
  static_assert(!F16S || (!FP16 && !MX), "fp16 scales serve bf16 activations");
  static_assert(!NV || (!MX && !F16S), "NVFP4 weights take 16-bit activations");
  constexpr int AB = MX ? 1 : 2;   // bytes per activation element the MMAs read
  constexpr int AIN = QA ? 2 : AB;  // bytes per activation element in HBM
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rg = warp;   // row group
  const int g = lane >> 2, t = lane & 3;
  const int S = p.splits;
  const int sl = blockIdx.x % S;   // rank in the cluster (clusters are S x 1 x 1)
  const int nt = blockIdx.x / S;
  const int kt0 = sl * p.kt / S, kt1 = (sl + 1) * p.kt / S;
  const int nk = kt1 - kt0;
  const int R = p.ring;
  const int BB = p.block_bytes;
  const int F = kTileN / S;        // features this CTA finishes
  // QA: act16 is the bf16 box, act the e4m3 tile quantized from it
  uint8_t* act16 = smem;
  uint8_t* act = QA ? smem + mma_act_bytes(p.nk_max, ROWS, 2) : smem;
  uint8_t* ring = act + mma_act_bytes(p.nk_max, ROWS, AB);
  float* recv = reinterpret_cast<float*>(ring + R * BB);          // [S][ROWS][F]
  float* amax_in = recv + ROWS * kTileN;          // QA: [S][ROWS] partial row maxima
  float* row_scale = amax_in + (QA ? 16 * ROWS : 0);   // QA: [ROWS]
  uint64_t* full = reinterpret_cast<uint64_t*>(row_scale + (QA ? ROWS : 0));
  uint64_t* empty = full + R;          // one arrival per warp when it is done with a slot
  uint64_t* act_full = empty + R;
  uint64_t* recv_full = act_full + 1;
  uint64_t* amax_full = recv_full + 1;   // QA: the S slices' maxima have landed
  int* issued = reinterpret_cast<int*>(amax_full + 1);   // weight blocks issued so far
  volatile int* abort_flag = issued + 1;
  const uint8_t* wsrc = p.w + ((long long)nt * p.kt + kt0) * BB;
  const int live = p.m < ROWS ? p.m : ROWS;
  // row r of the slice's activations at asrc + r * k * AIN
  const uint8_t* asrc = reinterpret_cast<const uint8_t*>(p.a) + (long long)kt0 * kTileK * AIN;

  if (tid == 0) {
    for (int s = 0; s < R; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kMmaWarps);
    }
    mbar_init(act_full, 1);
    mbar_init(recv_full, 1);
    mbar_init(amax_full, 1);
    fence_barrier_init();
    // the first weight blocks: issued before anything waits on the previous
    // grid (the slice's blocks, checked build: inside the layer's)
    const bool in = qg_check(nt < p.nt && kt0 >= 0 && kt1 <= p.kt, p.status);
    const int first = !in ? 0 : nk < R ? nk : R;
    const uint64_t pol = policy_evict_first();
    for (int s = 0; s < first; ++s) {
      mbar_arrive_expect_tx(&full[s], BB);
      bulk_load(ring + s * BB, wsrc + (long long)s * BB, BB, &full[s], pol);
    }
    *issued = first;
    *abort_flag = in ? 0 : 1;
    // the slices of the cluster's other CTAs (and this one's own) land here
    mbar_arrive_expect_tx(recv_full, (uint32_t)(S * live * F * 4));
    if constexpr (QA) mbar_arrive_expect_tx(amax_full, (uint32_t)(S * live * 4));
    prefetch_tmap(&tmap_a);
  }
  // the activation rows: an L2 prefetch now (the previous grid may still be
  // writing them; L2 is where its writes land, so a prefetched line is never
  // stale), the copy into shared memory after the wait
  if (warp == 1 && lane < live)
    prefetch_l2_bulk(asrc + (long long)lane * p.k * AIN, (uint32_t)(nk * kTileK * AIN));
  __syncthreads();
  cluster_sync_all();   // every receive barrier of the cluster is armed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) {
    // one box: nk_max k-tiles (AIN 128-byte chunks each) x ROWS rows (rows
    // past m and k past K read as zeros)
    mbar_arrive_expect_tx(act_full, (uint32_t)mma_act_bytes(p.nk_max, ROWS, AIN));
    tma_load_3d_hint(act16, &tmap_a, act_full, 0, 0, AIN * kt0, policy_evict_first());
  }

  float acc[2][2][NB][4];   // [k16 step parity][m16 block][n8 block]
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int c = 0; c < NB; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[h][b][c][i] = 0.f;

  constexpr uint32_t magic16 = FP16 ? 0x6400u : 0x4300u;
  // ldmatrix rows: lane l reads token (l & 7) + 8 (l >> 4) at k offset
  // 8 ((l >> 3) & 1); in the swizzled box, 16-byte unit u of row r of a chunk
  // sits at unit u ^ (r & 7)
  const int a_tok = (lane & 7) + 8 * (NB == 2 ? (lane >> 4) : 0);
  const uint32_t a_row = smem_u32(act) + (uint32_t)(a_tok * 128);
  const int a_x = a_tok & 7, a_k8 = (lane >> 3) & 1;
  bool ok = mbar_wait(act_full, 0, abort_flag, p.status, p.wait_limit_ns, kStatusTimeout);
  bool got_amax = true;
  if constexpr (QA) {
    // the slice's maximum |x| of each live row (the box may hold k-tiles of
    // the next slice or zeros past K: a maximum is unchanged by either), sent
    // to every CTA of the cluster (an aborted CTA sends too, so peers complete)
    const int units = 2 * p.nk_max * 8;   // 16-byte units of a row in the box
    for (int r = warp; r < live; r += kMmaWarps) {
      float mx_ = 0.f;
      for (int u = lane; u < units; u += 32) {
        const uint4 v = *reinterpret_cast<const uint4*>(act16 + (u >> 3) * (ROWS * 128) +
                                                        r * 128 + ((u & 7) << 4));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          mx_ = fmaxf(mx_, fmaxf(fabsf(__uint_as_float(w4[i] << 16)),
                                 fabsf(__uint_as_float(w4[i] & 0xFFFF0000u))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx_ = fmaxf(mx_, __shfl_xor_sync(0xffffffffu, mx_, o));
      if (lane < S) {
        const uint32_t dst = map_to_rank(smem_u32(amax_in + sl * ROWS + r), (uint32_t)lane);
        const uint32_t bar = map_to_rank(smem_u32(amax_full), (uint32_t)lane);
        asm volatile(
            "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(dst),
            "r"(__float_as_uint(mx_)), "r"(bar)
            : "memory");
      }
    }
    got_amax = mbar_wait(amax_full, 0, abort_flag, p.status, p.wait_limit_ns, kStatusTimeout);
    ok = ok && got_amax;
    // the rows' scales: the maximum over the S slices, then max / 448 (1 for
    // an all-zero row), an IEEE divide, as the standalone quantizer computes it
    if (tid < ROWS) {
      float s_ = 1.f;
      if (tid < live) {
        float a_ = 0.f;
        for (int q = 0; q < S; ++q) a_ = fmaxf(a_, amax_in[q * ROWS + tid]);
        s_ = a_ == 0.f ? 1.f : __fdiv_rn(a_, 448.f);
      }
      row_scale[tid] = s_;
    }
    __syncthreads();
    // e4m3 codes of the box: 16 k (two bf16 units, one e4m3 unit) per item;
    // rows past m stay zero
    const int items = ROWS * p.nk_max * 8;
    for (int i = tid; i < items; i += kMmaThreads) {
      const int r = i % ROWS, rest = i / ROWS, v8 = rest & 7, kt = rest >> 3;
      uint4 out = make_uint4(0u, 0u, 0u, 0u);
      if (r < live) {
        const float sc_ = row_scale[r];
        const uint8_t* c16 = act16 + (2 * kt + (v8 >> 2)) * (ROWS * 128) + r * 128;
        const int u0 = 2 * (v8 & 3);
        const uint4 x0 = *reinterpret_cast<const uint4*>(c16 + ((u0 ^ (r & 7)) << 4));
        const uint4 x1 = *reinterpret_cast<const uint4*>(c16 + (((u0 + 1) ^ (r & 7)) << 4));
        const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t ow[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint32_t hb = (xw[e >> 1] >> (16 * (e & 1))) << 16;
          const uint32_t code =
              __nv_cvt_float_to_fp8(__fdiv_rn(__uint_as_float(hb), sc_), __NV_SATFINITE,
                                    __NV_E4M3);
          ow[e >> 2] |= code << (8 * (e & 3));
        }
        out = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      }
      *reinterpret_cast<uint4*>(act + kt * (ROWS * 128) + r * 128 + ((v8 ^ (r & 7)) << 4)) =
          out;
    }
    __syncthreads();
  }
  int slot = 0;
  uint32_t phase = 0;
#pragma unroll 1
  for (int s = 0; s < nk && ok; ++s) {
    if (!mbar_wait(&full[slot], phase, abort_flag, p.status, p.wait_limit_ns, kStatusTimeout)) {
      ok = false;
      break;
    }
    const uint8_t* blk = ring + slot * BB;
    const uint4* wv = reinterpret_cast<const uint4*>(blk);
    if constexpr (MX) {
      // per row r: the four e8m0 scales of the k-tile's 32-k blocks (byte j)
      const uint32_t* sfw = reinterpret_cast<const uint32_t*>(blk + p.s_off);
      uint32_t sf[2][2];
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int e = 0; e < 2; ++e) sf[b][e] = sfw[rg * 32 + b * 16 + g + 8 * e];
      // the chunk (one per k-tile) of the e4m3 box; a 32-k block j is units
      // 2j (k 0-15: fragment b0) and 2j + 1 (k 16-31: b1)
      const uint32_t chunk = a_row + (uint32_t)(s * (ROWS * 128));
      const int sh = 16 * (t & 1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t bf[4];
        const uint32_t addr = chunk + (uint32_t)(((2 * j + a_k8) ^ a_x) * 16);
        if constexpr (NB == 2) {
          ldmatrix_x4(bf, addr);
        } else {
          uint32_t b2[2];
          ldmatrix_x2(b2, addr);
          bf[0] = b2[0];
          bf[1] = b2[1];
          bf[2] = bf[3] = 0u;
        }
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          // rows g, g + 8: the row's 32 codes, 16 bytes; lane t takes the codes
          // of k 4t..4t+3 (bytes 2t, 2t+1) and of k 16+4t.. (bytes 8+2t, 9+2t)
          const uint4 v0 = wv[(rg * 4 + j) * 32 + b * 16 + g];
          const uint4 v1 = wv[(rg * 4 + j) * 32 + b * 16 + g + 8];
          const uint32_t lo0 = (t & 2) ? v0.y : v0.x, hi0 = (t & 2) ? v0.w : v0.z;
          const uint32_t lo1 = (t & 2) ? v1.y : v1.x, hi1 = (t & 2) ? v1.w : v1.z;
          const uint32_t af[4] = {e2m1x4_e4m3(lo0 >> sh), e2m1x4_e4m3(lo1 >> sh),
                                  e2m1x4_e4m3(hi0 >> sh), e2m1x4_e4m3(hi1 >> sh)};
          const float s0 = e8m0_f32((sf[b][0] >> (8 * j)) & 0xFFu);
          const float s1 = e8m0_f32((sf[b][1] >> (8 * j)) & 0xFFu);
#pragma unroll
          for (int c = 0; c < NB; ++c) {
            float d[4];
            mma16832_e4m3(d, af, bf[2 * c], bf[2 * c + 1]);
            acc[j & 1][b][c][0] = fmaf(d[0], s0, acc[j & 1][b][c][0]);
            acc[j & 1][b][c][1] = fmaf(d[1], s0, acc[j & 1][b][c][1]);
            acc[j & 1][b][c][2] = fmaf(d[2], s1, acc[j & 1][b][c][2]);
            acc[j & 1][b][c][3] = fmaf(d[3], s1, acc[j & 1][b][c][3]);
          }
        }
      }
    } else {
    const uint16_t* sv = reinterpret_cast<const uint16_t*>(blk + p.s_off);
    const uint8_t* zv = blk + p.z_off;
    // per-row scale and zero pairs of rows (b, g) and (b, g + 8), group sg
    // (F16S: sc the scales' high bf16 terms, sl the low ones)
    [[maybe_unused]] uint32_t sl[2][2];
    auto row_consts = [&](int sg, uint32_t (&sc)[2][2], uint32_t (&zc)[2][2]) {
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = rg * 32 + b * 16 + g + 8 * e;
          if constexpr (F16S)
            split_f16_scale(sv[sg * kTileN + r], sc[b][e], sl[b][e]);
          else
            sc[b][e] = (uint32_t)sv[sg * kTileN + r] * 0x00010001u;
          zc[b][e] = (magic16 + (p.has_zp ? (uint32_t)zv[sg * kTileN + r] : 8u)) * 0x00010001u;
        }
    };
    uint32_t sc[2][2], zc[2][2];
    if constexpr (ONE_GROUP) row_consts(0, sc, zc);
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // 32-k chunk of the k-tile
      // B fragments of the chunk's two k16 steps: 64-k box chunk 2 s + j / 2,
      // 16-byte units 4 (j & 1) + 2 h + a_k8
      const uint32_t chunk = a_row + (uint32_t)((2 * s + (j >> 1)) * (ROWS * 128));
      uint32_t bf[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t addr = chunk + (uint32_t)((((4 * (j & 1) + 2 * h + a_k8) ^ a_x)) * 16);
        if constexpr (NB == 2) {
          ldmatrix_x4(bf[h], addr);
        } else {
          uint32_t b2[2];
          ldmatrix_x2(b2, addr);
          bf[h][0] = b2[0];
          bf[h][1] = b2[1];
          bf[h][2] = bf[h][3] = 0u;
        }
      }
      if constexpr (!ONE_GROUP && !NV) row_consts(j >> p.sg_shift, sc, zc);
      // m16 block b: rows 32 warp + 16 b + {g, g + 8} (e = 0, 1), 32 k each
      uint4 v[2][2];
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int e = 0; e < 2; ++e) v[b][e] = wv[(rg * 4 + j) * 32 + b * 16 + g + 8 * e];
      // A fragments of both blocks and both k16 steps, one stage at a time so
      // that the 16 independent chains interleave: fragment register i of
      // step h holds rows e = i & 1 of word 2h + (i >> 1) (k 8 (i >> 1) + 2t)
      uint32_t x[2][2][4];
      if constexpr (NV) {
        // block scales of rows (b, e): the 16-k blocks 2j + h of the k-tile
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const uint32_t s2 =
                  (uint32_t)sv[(2 * j + h) * kTileN + rg * 32 + b * 16 + g + 8 * e] * 0x00010001u;
              uint32_t c16, p0, p1;
              asm("prmt.b32 %0, %1, %2, %3;"
                  : "=r"(c16)
                  : "r"(word_of(v[b][e], 2 * h)), "r"(word_of(v[b][e], 2 * h + 1)),
                    "r"((uint32_t)(t | ((4 + t) << 4))));
              e2m1x4_pairs<FP16>(c16, p0, p1);
              x[b][h][e] = mul2<FP16>(p0, s2);
              x[b][h][2 + e] = mul2<FP16>(p1, s2);
            }
      } else {
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            x[b][h][i] = nib_pairs<FP16>(word_of(v[b][i & 1], 2 * h + (i >> 1)) >> (4 * t));
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 4; ++i) x[b][h][i] = sub2<FP16>(x[b][h][i], zc[b][i & 1]);
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if constexpr (F16S) {
              const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&x[b][h][i]);
              const __nv_bfloat162 r =
                  __hfma2(d, *reinterpret_cast<const __nv_bfloat162*>(&sc[b][i & 1]),
                          __hmul2(d, *reinterpret_cast<const __nv_bfloat162*>(&sl[b][i & 1])));
              x[b][h][i] = *reinterpret_cast<const uint32_t*>(&r);
            } else {
              x[b][h][i] = mul2<FP16>(x[b][h][i], sc[b][i & 1]);
            }
          }
      }   // integer codes
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          mma16816<FP16>(acc[h][b][0], x[b][h], bf[h][0], bf[h][1]);
          if constexpr (NB == 2) mma16816<FP16>(acc[h][b][1], x[b][h], bf[h][2], bf[h][3]);
        }
    }
    }   // 16-bit path
    // a ring shorter than the slice: every warp releases the slot, and warp
    // s % 4 refills it with block s + R once all four have
    if (R < nk) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if ((s & (kMmaWarps - 1)) == warp && s + R < nk) {
        if (lane == 0 &&
            mbar_wait(&empty[slot], phase, abort_flag, p.status, p.wait_limit_ns,
                      kStatusTimeout)) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&full[slot], BB);
          bulk_load(ring + slot * BB, wsrc + (long long)(s + R) * BB, BB, &full[slot],
                    policy_evict_first());
          atomicAdd(issued, 1);
        }
        __syncwarp();
      }
    }
    if (++slot == R) {
      slot = 0;
      phase ^= 1u;
    }
  }
  __syncthreads();   // every warp is done with the ring (and every refill issued)
  const bool aborted = *abort_flag != 0;
  if (aborted && tid == 0) {
    // let every copy this CTA issued land before shared memory is reused
    volatile int no_abort = 0;
    const int n_issued = *issued;
    for (int s = n_issued - R < 0 ? 0 : n_issued - R; s < n_issued; ++s)
      mbar_wait(&full[s % R], (uint32_t)((s / R) & 1), &no_abort, nullptr, kDrainLimitNs, 0);
    mbar_wait(act_full, 0, &no_abort, nullptr, kDrainLimitNs, 0);
    if (QA && !got_amax) mbar_wait(amax_full, 0, &no_abort, nullptr, kDrainLimitNs, 0);
  }
  __syncthreads();

  // the CTA's partial as [token][128 features] fp32 at the start of the ring
  float* part = reinterpret_cast<float*>(ring);
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      const int f = rg * 32 + b * 16 + g, tk = c * 8 + 2 * t;
      part[tk * kTileN + f] = acc[0][b][c][0] + acc[1][b][c][0];
      part[(tk + 1) * kTileN + f] = acc[0][b][c][1] + acc[1][b][c][1];
      part[tk * kTileN + f + 8] = acc[0][b][c][2] + acc[1][b][c][2];
      part[(tk + 1) * kTileN + f + 8] = acc[0][b][c][3] + acc[1][b][c][3];
    }
  __syncthreads();
  // push: features [r F, r F + F) of the live rows go to cluster rank r's
  // receive slot sl (an aborted CTA still sends, so every receiver completes)
  for (int i = tid; i < live * (kTileN / 4); i += kMmaThreads) {
    const int tk = i >> 5, f = (i & 31) * 4;
    const int r = f / F, off = f - r * F;
    const float4 v = *reinterpret_cast<const float4*>(part + tk * kTileN + f);
    const uint32_t dst = map_to_rank(smem_u32(recv + (sl * ROWS + tk) * F + off), (uint32_t)r);
    const uint32_t bar = map_to_rank(smem_u32(recv_full), (uint32_t)r);
    st_async_f4(dst, v, bar);
  }
  // finish features [sl F, sl F + F): the S slices summed in cluster-rank order
  const bool got = mbar_wait(recv_full, 0, abort_flag, p.status, p.wait_limit_ns, kStatusTimeout);
  if (!aborted && got) {
    const int q4 = F / 4;
    for (int i = tid; i < live * q4; i += kMmaThreads) {
      const int tk = i / q4, off = (i - tk * q4) * 4;
      float o[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < S; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(recv + (q * ROWS + tk) * F + off);
        o[0] += v.x;
        o[1] += v.y;
        o[2] += v.z;
        o[3] += v.w;
      }
      const int n = nt * kTileN + sl * F + off;
      if constexpr (MX) {   // the row's activation scale multiplies the fp32 sum
        const float as = QA ? row_scale[tk] : p.a_scale[tk];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] *= as;
      }
      if constexpr (NV) {   // the tensor scale multiplies the fp32 sum
        const float ts = p.t_scales[0];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] *= ts;
      }
      if (p.bias && qg_check(n + 4 <= p.n, p.status)) {
        const uint2 bb = *reinterpret_cast<const uint2*>(p.bias + n);
        const uint32_t bw[2] = {bb.x, bb.y};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint16_t h = (uint16_t)(bw[e >> 1] >> (16 * (e & 1)));
          o[e] += FP16 ? __half2float(__ushort_as_half(h))
                       : __bfloat162float(__ushort_as_bfloat16(h));
        }
      }
      uint32_t out[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if constexpr (FP16) {
          const __half2 h2 = __floats2half2_rn(o[2 * e], o[2 * e + 1]);
          out[e] = *reinterpret_cast<const uint32_t*>(&h2);
        } else {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * e], o[2 * e + 1]);
          out[e] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
      if (qg_check(tk < p.m && n + 4 <= p.n, p.status))
        *reinterpret_cast<uint2*>(p.c + (long long)tk * p.n + n) = make_uint2(out[0], out[1]);
    }
  }
  if (!got) {
    // every peer sends, so the slices arrive; a receiver that gave up still
    // waits (bounded) for them before its shared memory is released
    volatile int no_abort = 0;
    mbar_wait(recv_full, 0, &no_abort, nullptr, kDrainLimitNs, 0);
  }
}

template <bool FP16, int NB, bool ONE, bool MX = false, bool QA = false, bool F16S = false,
          bool NV = false>
static cudaError_t launch_one(const CUtensorMap& tmap, const W4A16MmaParams& p, int smem,
                              cudaStream_t stream) {
  auto kern = w4a16_mma_kernel<FP16, NB, ONE, MX, QA, F16S, NV>;
  static int smem_set = 0;
  static bool nonportable_set = false;
  if (smem > smem_set) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    smem_set = smem;
  }
  if (p.splits > 8 && !nonportable_set) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
    nonportable_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.nt * p.splits));
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)p.splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tmap, p);
}

cudaError_t launch_w4a16_mma(const CUtensorMap& tmap, const W4A16MmaParams& p, bool fp16,
                             cudaStream_t stream) {
  const bool one = p.sg_shift == 2;   // group >= 128
  const int nb = p.m <= 8 ? 1 : 2;
  const int smem =
      mma_smem_bytes(p.block_bytes, p.ring, p.nk_max, 8 * nb, p.mx ? 1 : 2, p.quant_act != 0);
  if (p.mx && p.quant_act)
    return nb == 1 ? launch_one<false, 1, true, true, true>(tmap, p, smem, stream)
                   : launch_one<false, 2, true, true, true>(tmap, p, smem, stream);
  if (p.mx)
    return nb == 1 ? launch_one<false, 1, true, true>(tmap, p, smem, stream)
                   : launch_one<false, 2, true, true>(tmap, p, smem, stream);
  if (p.nv) {
    if (fp16)
      return nb == 1 ? launch_one<true, 1, false, false, false, false, true>(tmap, p, smem, stream)
                     : launch_one<true, 2, false, false, false, false, true>(tmap, p, smem, stream);
    return nb == 1 ? launch_one<false, 1, false, false, false, false, true>(tmap, p, smem, stream)
                   : launch_one<false, 2, false, false, false, false, true>(tmap, p, smem, stream);
  }
  if (p.f16s) {
    if (nb == 1)
      return one ? launch_one<false, 1, true, false, false, true>(tmap, p, smem, stream)
                 : launch_one<false, 1, false, false, false, true>(tmap, p, smem, stream);
    return one ? launch_one<false, 2, true, false, false, true>(tmap, p, smem, stream)
               : launch_one<false, 2, false, false, false, true>(tmap, p, smem, stream);
  }
  if (fp16) {
    if (nb == 1) return one ? launch_one<true, 1, true>(tmap, p, smem, stream)
                            : launch_one<true, 1, false>(tmap, p, smem, stream);
    return one ? launch_one<true, 2, true>(tmap, p, smem, stream)
               : launch_one<true, 2, false>(tmap, p, smem, stream);
  }
  if (nb == 1) return one ? launch_one<false, 1, true>(tmap, p, smem, stream)
                          : launch_one<false, 1, false>(tmap, p, smem, stream);
  return one ? launch_one<false, 2, true>(tmap, p, smem, stream)
             : launch_one<false, 2, false>(tmap, p, smem, stream);
}

}  // namespace qg
