// Weight preprocessing: standard format -> the GEMM kernel's packed layout.
//
// The Humming preprocessing step checks parameters, pads dimensions and
// repacks tensors for the target kernel (kinachrichten.com, "Wie die
// Architektur funktioniert"); repacking rearranges without changing what the
// stored values mean (retrivium.ai, "vLLM Humming: why shared quantization
// still needs specialized kernels", section "Representation answers a
// different question").  Target layout (per expert; KT = K/128 k-tiles): one
// packed block per (n-tile, k-tile), n-tile major, so that the blocks of one
// n-tile's consecutive k-tiles are contiguous and a pipeline stage is filled
// by a single bulk copy.  A block is
//
//   codes    8192 bytes: 512 16-byte vectors, vector (qd*4 + j)*32 + t = row
//            32qd + t of the tile, k = 32j .. 32j+31.  INT4/UINT4: word w of
//            the vector holds 8 k, the nibble at position p holding k-offset
//            {0,2,4,6,1,3,5,7}[p], so a single 0x000F000F mask extracts two
//            consecutive k; INT4 codes are stored offset binary (q + 8).
//            MXFP4: the 16 bytes of the row's 32 codes in standard order.
//            INT8/UINT8: 16384 bytes, 1024 vectors, vector (qd*8 + j)*32 + t =
//            row 32qd + t, k = 16j .. 16j+15 in byte order; INT8 codes are
//            stored offset binary (q + 128).
//   scales   INT4/UINT4: 128 * ST 16-bit words (ST = max(1, 128/g)), word
//            sg*128 + r the scale of row r for the sg-th group of the tile.
//            MXFP4: 128 32-bit words, byte j of word r the e8m0 exponent of
//            row r for k = 32j .. 32j+31 of the tile.
//   zeros    UINT4 / UINT8 / UINT3 only: 128 * ST bytes, same order, the zero point.
//
// INT3 / UINT3 (GPTQ's 3-bit codes; the standard format is each column's
// codes as a little-endian bit stream along K, 32 codes in three words) are
// repacked into the 4-bit layout: an INT3 code q in [-4, 3] becomes the
// offset-binary nibble q + 8, exactly as an INT4 code does, and a UINT3 code
// and its zero point are stored as they are.  The 4-bit kernels then read
// them unchanged; every value means what the 3-bit code means.
//
// A gated layer's rows are taken in the gate/up interleaved order
// (glu_source_col).  Every thread writes one output vector / element; reads
// of the standard tensors are coalesced along N (in two runs per warp when
// gated).

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"

namespace qg {

__global__ void repack_weights_kernel(const int32_t* __restrict__ qweight, uint8_t* __restrict__ out,
                                      int n, int k, int signed_q, int block_bytes, int gated,
                                      long long total) {
  const long long vec = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (vec >= total) return;
  const int KT = k / kTileK, NT = n / kTileN;
  const long long per_expert = (long long)NT * KT * 512;
  const long long ex = vec / per_expert;
  const long long rem = vec - ex * per_expert;
  const long long blk = rem / 512;
  const int v = (int)(rem % 512);
  const int nt = (int)(blk / KT), kt = (int)(blk % KT);
  const int t = v & 31, j = (v >> 5) & 3, qd = v >> 7;
  const int col = packed_source_col(nt, qd * 32 + t, n, gated);
  const long long word_row0 = (long long)(kt * kTileK + j * 32) / 8;   // first K/8 row
  const int32_t* src = qweight + ex * (long long)(k / 8) * n;
  uint32_t o[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t in = (uint32_t)src[(word_row0 + w) * n + col];
    uint32_t r = 0;
    // nibble position p takes input nibble {0,2,4,6,1,3,5,7}[p]
    r |= ((in >> 0) & 0xFu) << 0;
    r |= ((in >> 8) & 0xFu) << 4;
    r |= ((in >> 16) & 0xFu) << 8;
    r |= ((in >> 24) & 0xFu) << 12;
    r |= ((in >> 4) & 0xFu) << 16;
    r |= ((in >> 12) & 0xFu) << 20;
    r |= ((in >> 20) & 0xFu) << 24;
    r |= ((in >> 28) & 0xFu) << 28;
    if (signed_q) r ^= 0x88888888u;   // two's complement nibble -> q + 8
    o[w] = r;
  }
  const long long gblk = ex * ((long long)NT * KT) + blk;
  *reinterpret_cast<uint4*>(out + gblk * block_bytes + v * 16) = make_uint4(o[0], o[1], o[2], o[3]);
}

// One thread per (block, group slot, row): the scale and (UINT4 / UINT8)
// the zero point; the codes take code_bytes at the start of each block.
__global__ void repack_scales_kernel(const uint16_t* __restrict__ scales,
                                     const int32_t* __restrict__ qzeros, uint8_t* __restrict__ out,
                                     int n, int k, int group, int block_bytes, int code_bytes,
                                     int zero_bits, int gated, long long total) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int KT = k / kTileK, NT = n / kTileN;
  const int st = group < kTileK ? kTileK / group : 1;
  const long long per_expert = (long long)NT * KT * st * kTileN;
  const long long ex = idx / per_expert;
  const long long rem = idx - ex * per_expert;
  const int r = (int)(rem % kTileN);
  const long long rest = rem / kTileN;
  const int sg = (int)(rest % st);
  const long long blk = rest / st;
  const int nt = (int)(blk / KT), kt = (int)(blk % KT);
  const int kk = kt * kTileK + sg * (group < kTileK ? group : kTileK);
  const int grp = kk / group;
  const int col = packed_source_col(nt, r, n, gated);
  const long long groups = k / group;
  uint8_t* bp = out + (ex * ((long long)NT * KT) + blk) * block_bytes;
  reinterpret_cast<uint16_t*>(bp + code_bytes)[sg * kTileN + r] =
      scales[ex * groups * n + (long long)grp * n + col];
  if (qzeros) {
    // the zero points of a group row are a little-endian bit stream along N:
    // column c's at bits [b c, b c + b), possibly straddling two words (b = 3)
    const long long row_words = (long long)n * zero_bits / 32;
    const int32_t* zr = qzeros + (ex * groups + grp) * row_words;
    const long long bit = (long long)zero_bits * col;
    const int off = (int)(bit & 31);
    uint64_t word = (uint32_t)zr[bit >> 5];
    if (off + zero_bits > 32) word |= (uint64_t)(uint32_t)zr[(bit >> 5) + 1] << 32;
    bp[code_bytes + packed_scale_bytes(false, st) + sg * kTileN + r] =
        (uint8_t)((word >> off) & ((1u << zero_bits) - 1u));
  }
}

// INT3 / UINT3 codes: output vector v of a block (row 32qd + t, k = 32j ..
// 32j + 31) takes the three standard words holding those 32 codes of the
// column (bits [3i, 3i + 3) of the 96-bit run for k = 32j + i) and writes
// them in the 4-bit vector's nibble order; INT3 codes become q + 8.
__global__ void repack_weights3_kernel(const int32_t* __restrict__ qweight,
                                       uint8_t* __restrict__ out, int n, int k, int signed_q,
                                       int block_bytes, int gated, long long total) {
  const long long vec = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (vec >= total) return;
  const int KT = k / kTileK, NT = n / kTileN;
  const long long per_expert = (long long)NT * KT * 512;
  const long long ex = vec / per_expert;
  const long long rem = vec - ex * per_expert;
  const long long blk = rem / 512;
  const int v = (int)(rem % 512);
  const int nt = (int)(blk / KT), kt = (int)(blk % KT);
  const int t = v & 31, j = (v >> 5) & 3, qd = v >> 7;
  const int col = packed_source_col(nt, qd * 32 + t, n, gated);
  const long long word_row0 = (long long)(kt * kTileK + j * 32) / 32 * 3;   // 3 words / 32 k
  const int32_t* src = qweight + ex * (long long)(k / 32 * 3) * n;
  const uint32_t w0 = (uint32_t)src[(word_row0 + 0) * n + col];
  const uint32_t w1 = (uint32_t)src[(word_row0 + 1) * n + col];
  const uint32_t w2 = (uint32_t)src[(word_row0 + 2) * n + col];
  auto code = [&](int i) -> uint32_t {   // the 3-bit code of k = 32j + i
    const int b = 3 * i;
    uint64_t x = b < 32 ? ((uint64_t)w0 | ((uint64_t)w1 << 32)) >> b
                        : ((uint64_t)w1 | ((uint64_t)w2 << 32)) >> (b - 32);
    const uint32_t c = (uint32_t)x & 7u;
    // two's complement q = c - 8 [c >= 4] -> q + 8 = (c ^ 4) + 4
    return signed_q ? (c ^ 4u) + 4u : c;
  };
  uint32_t o[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    // nibble position p takes k-offset {0,2,4,6,1,3,5,7}[p] of the word's 8 k
    uint32_t r = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int koff = p < 4 ? 2 * p : 2 * (p - 4) + 1;
      r |= code(8 * w + koff) << (4 * p);
    }
    o[w] = r;
  }
  const long long gblk = ex * ((long long)NT * KT) + blk;
  *reinterpret_cast<uint4*>(out + gblk * block_bytes + v * 16) = make_uint4(o[0], o[1], o[2], o[3]);
}

// INT8 / UINT8 codes: output vector v of a block takes four standard words
// (16 consecutive k of one column) unchanged in byte order; INT8 bytes move
// to offset binary.
__global__ void repack_weights8_kernel(const int32_t* __restrict__ qweight,
                                       uint8_t* __restrict__ out, int n, int k, int signed_q,
                                       int block_bytes, int gated, long long total) {
  const long long vec = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (vec >= total) return;
  const int KT = k / kTileK, NT = n / kTileN;
  const long long per_expert = (long long)NT * KT * 1024;
  const long long ex = vec / per_expert;
  const long long rem = vec - ex * per_expert;
  const long long blk = rem / 1024;
  const int v = (int)(rem % 1024);
  const int nt = (int)(blk / KT), kt = (int)(blk % KT);
  const int t = v & 31, j = (v >> 5) & 7, qd = v >> 8;
  const int col = packed_source_col(nt, qd * 32 + t, n, gated);
  const long long word_row0 = (long long)(kt * kTileK + j * 16) / 4;   // first K/4 row
  const int32_t* src = qweight + ex * (long long)(k / 4) * n;
  uint32_t o[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t in = (uint32_t)src[(word_row0 + w) * n + col];
    o[w] = signed_q ? in ^ 0x80808080u : in;   // two's complement byte -> q + 128
  }
  const long long gblk = ex * ((long long)NT * KT) + blk;
  *reinterpret_cast<uint4*>(out + gblk * block_bytes + v * 16) = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaError_t launch_repack_w4(const int32_t* qweight, const uint16_t* scales,
                             const int32_t* qzeros, uint8_t* packed, int64_t n, int64_t k,
                             int group, int signed_q, int experts, int gated, int code_bits,
                             cudaStream_t stream) {
  const int threads = 256;
  const int st = group < kTileK ? kTileK / group : 1;
  const int block_bytes = packed_block_bytes(false, st, qzeros != nullptr);
  const long long vecs = (long long)experts * (n / kTileN) * (k / kTileK) * 512;
  if (code_bits == 3)
    repack_weights3_kernel<<<(unsigned)((vecs + threads - 1) / threads), threads, 0, stream>>>(
        qweight, packed, (int)n, (int)k, signed_q, block_bytes, gated, vecs);
  else
    repack_weights_kernel<<<(unsigned)((vecs + threads - 1) / threads), threads, 0, stream>>>(
        qweight, packed, (int)n, (int)k, signed_q, block_bytes, gated, vecs);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const long long elems = (long long)experts * (n / kTileN) * (k / kTileK) * st * kTileN;
  repack_scales_kernel<<<(unsigned)((elems + threads - 1) / threads), threads, 0, stream>>>(
      scales, qzeros, packed, (int)n, (int)k, group, block_bytes, packed_code_bytes(false),
      code_bits, gated, elems);
  return cudaGetLastError();
}

cudaError_t launch_repack_w8(const int32_t* qweight, const uint16_t* scales,
                             const int32_t* qzeros, uint8_t* packed, int64_t n, int64_t k,
                             int group, int signed_q, int experts, int gated,
                             cudaStream_t stream) {
  const int threads = 256;
  const int st = group < kTileK ? kTileK / group : 1;
  const int block_bytes = packed_block_bytes(false, st, qzeros != nullptr, true);
  const long long vecs = (long long)experts * (n / kTileN) * (k / kTileK) * 1024;
  repack_weights8_kernel<<<(unsigned)((vecs + threads - 1) / threads), threads, 0, stream>>>(
      qweight, packed, (int)n, (int)k, signed_q, block_bytes, gated, vecs);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const long long elems = (long long)experts * (n / kTileN) * (k / kTileK) * st * kTileN;
  repack_scales_kernel<<<(unsigned)((elems + threads - 1) / threads), threads, 0, stream>>>(
      scales, qzeros, packed, (int)n, (int)k, group, block_bytes, packed_code_bytes(true), 8,
      gated, elems);
  return cudaGetLastError();
}

// MXFP4: standard codes [N, K/2] (k = 2j low nibble, 2j+1 high nibble) and
// e8m0 scales [N, K/32] -> packed blocks (layout above); the nibbles stay in
// their standard order because the kernel's table lookup wants consecutive k
// in consecutive nibbles.
__global__ void repack_mxfp4_kernel(const uint8_t* __restrict__ codes,
                                    const uint8_t* __restrict__ scales, uint8_t* __restrict__ out,
                                    int n, int k, int gated, long long vecs, long long words) {
  constexpr int kBlock = packed_block_bytes(true, 1, false);
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int KT = k / kTileK, NT = n / kTileN;
  if (idx < vecs) {
    const long long per_expert = (long long)NT * KT * 512;
    const long long ex = idx / per_expert;
    const long long rem = idx - ex * per_expert;
    const long long blk = rem / 512;
    const int v = (int)(rem % 512);
    const int nt = (int)(blk / KT), kt = (int)(blk % KT);
    const int t = v & 31, j = (v >> 5) & 3, qd = v >> 7;
    const long long row = packed_source_col(nt, qd * 32 + t, n, gated);
    const uint8_t* src = codes + (ex * n + row) * (k / 2) + (kt * kTileK + j * 32) / 2;
    *reinterpret_cast<uint4*>(out + (ex * ((long long)NT * KT) + blk) * kBlock + v * 16) =
        *reinterpret_cast<const uint4*>(src);
  }
  if (idx < words) {
    const long long per_expert = (long long)NT * KT * kTileN;
    const long long ex = idx / per_expert;
    const long long rem = idx - ex * per_expert;
    const int r = (int)(rem % kTileN);
    const long long blk = rem / kTileN;
    const int nt = (int)(blk / KT), kt = (int)(blk % KT);
    const long long row = packed_source_col(nt, r, n, gated);
    reinterpret_cast<uint32_t*>(out + (ex * ((long long)NT * KT) + blk) * kBlock + kTileBytes)[r] =
        *reinterpret_cast<const uint32_t*>(scales + (ex * n + row) * (k / 32) + kt * 4);
  }
}

cudaError_t launch_repack_mxfp4(const uint8_t* codes, const uint8_t* scales, uint8_t* packed,
                                int64_t n, int64_t k, int experts, int gated,
                                cudaStream_t stream) {
  const long long tiles = (long long)experts * (n / kTileN) * (k / kTileK);
  const long long vecs = tiles * 512, words = tiles * kTileN;
  const long long total = vecs > words ? vecs : words;
  const int threads = 256;
  repack_mxfp4_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, stream>>>(
      codes, scales, packed, (int)n, (int)k, gated, vecs, words);
  return cudaGetLastError();
}

// NVFP4: standard codes [N, K/2] (as MXFP4) and e4m3 block scales [N, K/16]
// -> packed blocks: the code vectors exactly as MXFP4's, the block scales as
// the activation dtype's 16-bit pattern of the same value (every e4m3 value is
// a bf16 and an fp16 value) at word sg * 128 + r, sg the 16-k group within the
// k-tile; the per-expert fp32 tensor scales follow the last block.
__global__ void repack_nvfp4_kernel(const uint8_t* __restrict__ codes,
                                    const uint8_t* __restrict__ scales,
                                    const float* __restrict__ tensor_scales,
                                    uint8_t* __restrict__ out, int n, int k, int experts, int fp16,
                                    int gated, long long vecs, long long words) {
  constexpr int kBlock = packed_block_bytes(false, 8, false);
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int KT = k / kTileK, NT = n / kTileN;
  if (idx < vecs) {
    const long long per_expert = (long long)NT * KT * 512;
    const long long ex = idx / per_expert;
    const long long rem = idx - ex * per_expert;
    const long long blk = rem / 512;
    const int v = (int)(rem % 512);
    const int nt = (int)(blk / KT), kt = (int)(blk % KT);
    const int t = v & 31, j = (v >> 5) & 3, qd = v >> 7;
    const long long row = packed_source_col(nt, qd * 32 + t, n, gated);
    const uint8_t* src = codes + (ex * n + row) * (k / 2) + (kt * kTileK + j * 32) / 2;
    *reinterpret_cast<uint4*>(out + (ex * ((long long)NT * KT) + blk) * kBlock + v * 16) =
        *reinterpret_cast<const uint4*>(src);
  }
  if (idx < words) {
    const long long per_expert = (long long)NT * KT * 8 * kTileN;
    const long long ex = idx / per_expert;
    const long long rem = idx - ex * per_expert;
    const int r = (int)(rem % kTileN);
    const long long rest = rem / kTileN;
    const int sg = (int)(rest % 8);
    const long long blk = rest / 8;
    const int nt = (int)(blk / KT), kt = (int)(blk % KT);
    const long long row = packed_source_col(nt, r, n, gated);
    const uint8_t e4 = scales[(ex * n + row) * (k / 16) + kt * 8 + sg];
    const __half_raw hr = __nv_cvt_fp8_to_halfraw(e4, __NV_E4M3);
    uint16_t bits = hr.x;
    if (!fp16) {
      const __nv_bfloat16 b = __float2bfloat16_rn(__half2float(__half(hr)));   // exact
      bits = *reinterpret_cast<const uint16_t*>(&b);
    }
    reinterpret_cast<uint16_t*>(out + (ex * ((long long)NT * KT) + blk) * kBlock +
                                kTileBytes)[sg * kTileN + r] = bits;
  }
  if (idx < ((experts + 3) & ~3)) {   // the tail, zero-padded to 16 bytes
    float* tail = reinterpret_cast<float*>(out + (long long)experts * NT * KT * kBlock);
    tail[idx] = idx < experts ? tensor_scales[idx] : 0.f;
  }
}

cudaError_t launch_repack_nvfp4(const uint8_t* codes, const uint8_t* scales,
                               const float* tensor_scales, uint8_t* packed, int64_t n, int64_t k,
                               int experts, bool fp16, int gated, cudaStream_t stream) {
  const long long tiles = (long long)experts * (n / kTileN) * (k / kTileK);
  const long long vecs = tiles * 512, words = tiles * 8 * kTileN;
  long long total = vecs > words ? vecs : words;
  if (total < ((experts + 3) & ~3)) total = (experts + 3) & ~3;
  const int threads = 256;
  repack_nvfp4_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, stream>>>(
      codes, scales, tensor_scales, packed, (int)n, (int)k, experts, fp16 ? 1 : 0, gated, vecs,
      words);
  return cudaGetLastError();
}

}  // namespace qg
