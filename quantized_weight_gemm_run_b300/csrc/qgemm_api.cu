// The C ABI (include/qgemm.h): validation, the B300 tuning heuristic, plans,
// tensor maps and launches.  Host code only; the kernels live in the other
// translation units.
//
// The three-config split (layer / compute / tuning), the device heuristic
// that picks a tuning per input-size range, and the explicit rejection of
// unsupported combinations follow the Humming pages (kinachrichten.com,
// "Wie die Architektur funktioniert"; retrivium.ai, "vLLM Humming: why
// shared quantization still needs specialized kernels", section "The
// architectural gain is a smaller maintenance surface").  The plan record
// written by qgemm_describe_plan follows the compatibility record of the
// retrivium.ai retrospective on the format-kernel contract (section "A
// compatibility example"): representation, activation type, device and shape,
// and which implementation serves them.

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/qgemm.h"
#include "internal.h"

namespace qg {

static thread_local std::string g_last_error;
static unsigned long long g_wait_limit_ns = 1000000000ull;

static qgemm_status fail(qgemm_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

static qgemm_status ok() {
  g_last_error.clear();
  return QGEMM_OK;
}

static qgemm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(QGEMM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device properties, queried once per device (up to 64 devices).
struct DeviceProps {
  int sms = 0, max_smem = 0, major = 0, minor = 0;
};

static const DeviceProps* device_props() {
  static DeviceProps props[64];
  static std::once_flag once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::call_once(once[dev], [dev] {
    DeviceProps& d = props[dev];
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
  });
  return props[dev].sms > 0 ? &props[dev] : nullptr;
}

int device_sm_count() {
  const DeviceProps* d = device_props();
  return d ? d->sms : 0;
}

static int device_max_smem() {
  const DeviceProps* d = device_props();
  return d ? d->max_smem : 0;
}

static bool device_is_sm103() {
  const DeviceProps* d = device_props();
  return d && d->major == 10 && d->minor == 3;
}

// ------------------------------------------------------------ validation

static qgemm_status check_layer(const qgemm_layer_config* L) {
  if (!L) return fail(QGEMM_ERR_INVALID_ARG, "layer config is NULL");
  if (L->n <= 0 || L->k <= 0) return fail(QGEMM_ERR_INVALID_ARG, "n and k must be positive");
  if (L->num_experts < 1) return fail(QGEMM_ERR_INVALID_ARG, "num_experts must be >= 1");
  if (L->num_experts > kMaxExperts)
    return fail(QGEMM_ERR_UNSUPPORTED, "num_experts %d exceeds %d", L->num_experts, kMaxExperts);
  if (L->n % kTileN || L->k % kTileK)
    return fail(QGEMM_ERR_UNSUPPORTED, "n and k must be multiples of 128 (got n=%lld k=%lld)",
                (long long)L->n, (long long)L->k);
  if (L->n > (1 << 20) || L->k > (1 << 20))
    return fail(QGEMM_ERR_UNSUPPORTED, "n or k above 2^20");
  if (L->has_bias != 0 && L->has_bias != 1)
    return fail(QGEMM_ERR_INVALID_ARG, "has_bias must be 0 or 1");
  if (L->gated_act != QGEMM_ACT_NONE && L->gated_act != QGEMM_ACT_SILU_GLU)
    return fail(QGEMM_ERR_INVALID_ARG, "unknown gated_act %d", L->gated_act);
  if (L->gated_act != QGEMM_ACT_NONE && L->out_dtype != QGEMM_BF16)
    return fail(QGEMM_ERR_UNSUPPORTED, "a gated output must be bf16");
  switch (L->weight_format) {
    case QGEMM_W_INT3_SYM:
    case QGEMM_W_UINT3_ZP:
    case QGEMM_W_INT4_SYM:
    case QGEMM_W_UINT4_ZP: {
      const bool w3 = L->weight_format == QGEMM_W_INT3_SYM || L->weight_format == QGEMM_W_UINT3_ZP;
      const bool sym = L->weight_format == QGEMM_W_INT4_SYM || L->weight_format == QGEMM_W_INT3_SYM;
      if (L->act_dtype != QGEMM_FP16 && L->act_dtype != QGEMM_BF16)
        return fail(QGEMM_ERR_UNSUPPORTED, "W4A16 needs fp16 or bf16 activations");
      if (L->out_dtype != L->act_dtype)
        return fail(QGEMM_ERR_UNSUPPORTED, "W4A16 output dtype must equal the activation dtype");
      if (L->scale_format != QGEMM_S_FP16 && L->scale_format != QGEMM_S_BF16)
        return fail(QGEMM_ERR_UNSUPPORTED, "W4A16 scales must be fp16 or bf16");
      if (L->scale_format == QGEMM_S_BF16 && L->act_dtype == QGEMM_FP16)
        return fail(QGEMM_ERR_UNSUPPORTED, "bf16 scales need bf16 activations");
      const int g = L->group_size;
      const bool g_ok = g == 32 || g == 64 || (g >= 128 && g % 128 == 0);
      if (!g_ok) return fail(QGEMM_ERR_UNSUPPORTED, "group size %d not in {32, 64, 128j}", g);
      if (L->k % g) return fail(QGEMM_ERR_UNSUPPORTED, "k must be a multiple of the group size");
      if (sym && L->zero_format != QGEMM_Z_NONE)
        return fail(QGEMM_ERR_UNSUPPORTED, "symmetric integer weights take no zero points");
      if (!sym && L->zero_format != (w3 ? QGEMM_Z_UINT3 : QGEMM_Z_UINT4))
        return fail(QGEMM_ERR_UNSUPPORTED, w3 ? "UINT3 needs uint3 zero points"
                                                : "UINT4 needs uint4 zero points");
      return ok();
    }
    case QGEMM_W_INT8_SYM:
    case QGEMM_W_UINT8_ZP: {
      if (L->act_dtype != QGEMM_FP16 && L->act_dtype != QGEMM_BF16)
        return fail(QGEMM_ERR_UNSUPPORTED, "W8A16 needs fp16 or bf16 activations");
      if (L->out_dtype != L->act_dtype)
        return fail(QGEMM_ERR_UNSUPPORTED, "W8A16 output dtype must equal the activation dtype");
      if ((L->scale_format == QGEMM_S_FP16 ? QGEMM_FP16 : L->scale_format == QGEMM_S_BF16
                                                              ? QGEMM_BF16
                                                              : -1) != L->act_dtype)
        return fail(QGEMM_ERR_UNSUPPORTED, "W8A16 scales must be in the activation dtype");
      const int g = L->group_size;
      if (!(g == 32 || g == 64 || (g >= 128 && g % 128 == 0)))
        return fail(QGEMM_ERR_UNSUPPORTED, "group size %d not in {32, 64, 128j}", g);
      if (L->k % g) return fail(QGEMM_ERR_UNSUPPORTED, "k must be a multiple of the group size");
      if (L->weight_format == QGEMM_W_INT8_SYM && L->zero_format != QGEMM_Z_NONE)
        return fail(QGEMM_ERR_UNSUPPORTED, "symmetric INT8 takes no zero points");
      if (L->weight_format == QGEMM_W_UINT8_ZP && L->zero_format != QGEMM_Z_UINT8)
        return fail(QGEMM_ERR_UNSUPPORTED, "UINT8 needs uint8 zero points");
      return ok();
    }
    case QGEMM_W_NVFP4:
      if (L->zero_format != QGEMM_Z_NONE)
        return fail(QGEMM_ERR_UNSUPPORTED, "NVFP4 takes no zero points");
      if (L->scale_format != QGEMM_S_E4M3 || L->group_size != 16)
        return fail(QGEMM_ERR_UNSUPPORTED, "NVFP4 needs e4m3 scales per 16 k");
      if (L->act_dtype == QGEMM_NVFP4) {   // W4A4
        if (L->out_dtype != QGEMM_BF16)
          return fail(QGEMM_ERR_UNSUPPORTED, "W4A4 writes a bf16 output");
        if (L->k % kW4A4TileK)
          return fail(QGEMM_ERR_UNSUPPORTED, "W4A4 needs k a multiple of 256");
        if (L->num_experts != 1 || L->gated_act != QGEMM_ACT_NONE)
          return fail(QGEMM_ERR_UNSUPPORTED, "W4A4 runs dense, ungated GEMMs");
        return ok();
      }
      if (L->act_dtype != QGEMM_FP16 && L->act_dtype != QGEMM_BF16)
        return fail(QGEMM_ERR_UNSUPPORTED, "NVFP4 weights run against fp16 or bf16 activations");
      if (L->out_dtype != L->act_dtype)
        return fail(QGEMM_ERR_UNSUPPORTED, "the output dtype must equal the activation dtype");
      return ok();
    case QGEMM_W_MXFP4:
      if (L->zero_format != QGEMM_Z_NONE)
        return fail(QGEMM_ERR_UNSUPPORTED, "MXFP4 takes no zero points");
      if (L->scale_format != QGEMM_S_E8M0 || L->group_size != 32)
        return fail(QGEMM_ERR_UNSUPPORTED, "MXFP4 needs e8m0 scales per 32 k");
      // e4m3 activations with the caller's per-row scales, or bf16 ones that
      // the library quantizes per row
      if ((L->act_dtype != QGEMM_FP8E4M3 && L->act_dtype != QGEMM_BF16) ||
          L->out_dtype != QGEMM_BF16)
        return fail(QGEMM_ERR_UNSUPPORTED,
                    "MXFP4 runs against e4m3 or bf16 activations, bf16 output");
      return ok();
    default:
      return fail(QGEMM_ERR_UNSUPPORTED, "unknown weight format %d", L->weight_format);
  }
}

static qgemm_status check_compute(const qgemm_compute_config* C, const qgemm_layer_config* L,
                                  bool grouped_call) {
  if (!C) return fail(QGEMM_ERR_INVALID_ARG, "compute config is NULL");
  if (C->batch_invariant != 0 && C->batch_invariant != 1)
    return fail(QGEMM_ERR_INVALID_ARG, "batch_invariant must be 0 or 1");
  if (C->deterministic != 0 && C->deterministic != 1)
    return fail(QGEMM_ERR_INVALID_ARG, "deterministic must be 0 or 1");
  if (C->gemm_type != (grouped_call ? QGEMM_GEMM_GROUPED : QGEMM_GEMM_DENSE))
    return fail(QGEMM_ERR_INVALID_ARG, "gemm_type does not match the entry point");
  if (!grouped_call && L->num_experts != 1)
    return fail(QGEMM_ERR_INVALID_ARG, "a dense GEMM needs num_experts = 1");
  return ok();
}

static int st_of(int group) { return group < kTileK ? kTileK / group : 1; }

static bool is_mx(const qgemm_layer_config* L) { return L->weight_format == QGEMM_W_MXFP4; }
static bool is_nv(const qgemm_layer_config* L) { return L->weight_format == QGEMM_W_NVFP4; }
// W4A4: NVFP4 weights against activations the library quantizes to NVFP4
static bool is_w4a4(const qgemm_layer_config* L) {
  return is_nv(L) && L->act_dtype == QGEMM_NVFP4;
}
// W4A8 whose bf16 activations the library quantizes per row to e4m3
static bool quant_in_lib(const qgemm_layer_config* L) {
  return is_mx(L) && L->act_dtype == QGEMM_BF16;
}
static bool is_w8(const qgemm_layer_config* L) {
  return L->weight_format == QGEMM_W_INT8_SYM || L->weight_format == QGEMM_W_UINT8_ZP;
}
// integer formats with zero points (UINT4, UINT8)
static bool has_zeros(const qgemm_layer_config* L) {
  return L->zero_format == QGEMM_Z_UINT4 || L->zero_format == QGEMM_Z_UINT8 ||
         L->zero_format == QGEMM_Z_UINT3;
}
// 3-bit integer codes (GPTQ INT3 / UINT3), repacked into the 4-bit blocks
static bool is_w3(const qgemm_layer_config* L) {
  return L->weight_format == QGEMM_W_INT3_SYM || L->weight_format == QGEMM_W_UINT3_ZP;
}
// W4A16 with fp16 scales against bf16 activations
static bool is_f16s(const qgemm_layer_config* L) {
  return !is_mx(L) && !is_nv(L) && !is_w8(L) && L->scale_format == QGEMM_S_FP16 &&
         L->act_dtype == QGEMM_BF16;
}

// The tcgen05 kernel's format instantiation (see launch_w4a16).
static int fmt_of(const qgemm_layer_config* L) {
  const bool fp16 = L->act_dtype == QGEMM_FP16;
  if (is_mx(L)) return 2;
  if (is_nv(L)) return fp16 ? 4 : 3;
  if (is_f16s(L)) return 5;
  if (is_w8(L)) return fp16 ? 7 : 6;
  return fp16 ? 1 : 0;
}

// Bytes of one expert's packed blocks (an NVFP4 buffer adds the tensor-scale
// tail after the last expert).
static size_t expert_packed_bytes(const qgemm_layer_config* L) {
  const size_t tiles = (size_t)(L->n / kTileN) * (size_t)(L->k / kTileK);
  return tiles * (size_t)packed_block_bytes(is_mx(L), st_of(L->group_size), has_zeros(L),
                                            is_w8(L));
}

// ------------------------------------------------------------ plans

WorkspaceLayout workspace_layout(int64_t max_tiles, int grid, int block_tok) {
  WorkspaceLayout w;
  w.counters_off = 256;
  w.counters_bytes = ((size_t)max_tiles * 4 * sizeof(int) + 255) & ~size_t(255);
  w.partials_off = w.counters_off + w.counters_bytes;
  w.partials_bytes = (size_t)2 * grid * block_tok * kTileN * sizeof(float);
  w.total = w.partials_off + w.partials_bytes;
  w.aq_off = w.aq_scale_off = w.total;
  w.aq_bytes = 0;
  return w;
}

// Appends the region of the library-quantized activations (rows x k e4m3
// codes, then rows fp32 scales).
static void add_act_quant_region(WorkspaceLayout* w, int64_t rows, int64_t k) {
  const size_t codes = ((size_t)rows * (size_t)k + 255) & ~size_t(255);
  const size_t scales = ((size_t)rows * sizeof(float) + 255) & ~size_t(255);
  w->aq_off = w->total;
  w->aq_scale_off = w->aq_off + codes;
  w->aq_bytes = codes + scales;
  w->total += w->aq_bytes;
}

static int heuristic_block_tok(int64_t rows_per_group) {
  if (rows_per_group <= 16) return 16;
  if (rows_per_group <= 32) return 32;
  if (rows_per_group <= 64) return 64;
  return 128;
}

// Shared-memory geometry: the activation ring (1 KB aligned slots of
// units_per_stage(bt) token tiles), the weight ring (slots of
// weight_units_per_slot(bt) packed blocks), the per-warp output staging
// buffers, then barriers, shared state and the grouped prefix arrays.  The
// activation ring gets enough slots to cover a copy's latency at the tensor
// rate; the weight ring gets the rest of shared memory (at most w_cap slots),
// since it is what streams from HBM at small M.
// A cluster-split launch adds the receive slots of the other slices
// (recv_bytes) after the staging buffers.
struct Geometry {
  int x_bytes, x_stages, w_bytes, w_stages, rw, off_w, off_epi, off_recv, off_bar, smem;
};

static int tail_smem(int sx, int sw, int experts) {
  return (2 * sx + 2 * sw + 2 * kASlots + 4 + 2 + 4 + 1) * 8 + 32 + 2 * (experts + 1) * 4 + 64;
}

static bool make_geometry(int bt, int st, int has_zp, bool mx, bool w8, int experts, int w_cap,
                          int smem_cap, int recv_bytes, Geometry* g) {
  const int rx = units_per_stage(bt);
  g->rw = weight_units_per_slot(bt);
  g->x_bytes = (rx * bt * kTileK * (mx ? 1 : 2) + 1023) & ~1023;
  g->w_bytes = g->rw * packed_block_bytes(mx, st, has_zp != 0, w8);
  for (int sx = bt <= 32 ? 3 : 4; sx >= 2; --sx) {
    const int fixed = 1024 /* alignment slack */ + sx * g->x_bytes + 1023 + kEpiStageBytes +
                      recv_bytes + tail_smem(sx, 16, experts);
    int sw = (smem_cap - fixed) / g->w_bytes;
    if (sw > w_cap) sw = w_cap;
    if (sw < 2) continue;
    g->x_stages = sx;
    g->w_stages = sw;
    g->off_w = sx * g->x_bytes;
    g->off_epi = (g->off_w + sw * g->w_bytes + 1023) & ~1023;
    g->off_recv = g->off_epi + kEpiStageBytes;
    g->off_bar = g->off_recv + recv_bytes;
    g->smem = 1024 + g->off_bar + tail_smem(sx, sw, experts);
    if (g->smem <= smem_cap) return true;
  }
  return false;
}

struct Plan {
  int kernel;        // 1: the persistent tcgen05 kernel, 2: the small-M mma.sync kernel
  int mma_splits;    // small-M kernel: K slices per n-tile (CTAs per cluster)
  int mma_ring;      // small-M kernel: weight slots per CTA
  int mma_nk_max;    // small-M kernel: most k-tiles in one slice
  int bt, grid, st, off_s, off_z;
  int split_cap;     // most CTAs sharing one tile's K range (0: no cap, 1: whole tiles)
  int cluster;       // tcgen05 kernel: S > 1 = cluster split of S CTAs per tile, else 0
  Geometry g;
  int64_t max_tiles;
  WorkspaceLayout ws;
};

// C may be null (the default compute config).
static qgemm_status make_plan(const qgemm_layer_config* L, const qgemm_tuning_config* T,
                              const qgemm_compute_config* C, int64_t rows, bool grouped,
                              Plan* P) {
  *P = Plan();
  // most CTAs per tile: from the tuning; 1 (whole tiles) under batch
  // invariance, since a split's K boundaries depend on the tile count (so on M)
  int cap = T ? T->split_k : 0;
  if (C && C->batch_invariant == 1) cap = 1;
  const int sms = device_sm_count();
  if (sms <= 0) return fail(QGEMM_ERR_CUDA, "no CUDA device");
  const int E = L->num_experts;
  // Grouped: expert row counts scatter around the mean, and a tile shorter
  // than an expert's rows dequantizes that expert's weights once per tile, so
  // the tile is sized for 1.5 x the mean (measured on B300, E = 64, top-8,
  // hidden 2048, T = 256: 64-token tiles 128-131 us against 150-152 us with
  // 32; T = 16 and 4096 keep 16 and 128)
  int bt = (T && T->block_tok) ? T->block_tok
                               : heuristic_block_tok(grouped ? (3 * rows + 2 * E - 1) / (2 * E)
                                                             : rows);
  // W4A8 (measured on B300, N = 7168, K = 2048, M = 128): 64-token whole tiles
  // in one wave beat 128-token tiles when they fit (13.2 against 15.3 us)
  if (is_mx(L) && !grouped && !(T && T->block_tok) && bt == 128 &&
      ((rows + 63) / 64) * (L->n / kTileN) <= device_sm_count())
    bt = 64;
  if (bt != 16 && bt != 32 && bt != 64 && bt != 128 && bt != 256)
    return fail(QGEMM_ERR_UNSUPPORTED, "block_tok %d not in {16, 32, 64, 128, 256}", bt);
  if (bt == 256 && (is_mx(L) || is_nv(L) || is_f16s(L) || is_w8(L)))
    return fail(QGEMM_ERR_UNSUPPORTED,
                "block_tok 256 takes INT4 / UINT4 weights with scales in the activation dtype");
  if (T && (T->cta_pair != 0)) return fail(QGEMM_ERR_UNSUPPORTED, "cta_pair is reserved");
  if (T && (T->split_k < 0 || T->split_k > 64))
    return fail(QGEMM_ERR_INVALID_ARG, "split_k must be in [0, 64]");
  const int st = st_of(L->group_size);
  const int has_zp = has_zeros(L);
  if (T && (T->kernel < 0 || T->kernel > 3))
    return fail(QGEMM_ERR_INVALID_ARG, "kernel must be 0, 1, 2 or 3");
  const int64_t ntl = L->n / kTileN, ktl = L->k / kTileK;
  // small-M kernel: K slices per n-tile (a power of two, at most 16 and at
  // most the k-tiles), and weight slots per CTA
  int64_t S = 0;
  if (T && T->kernel == 2 && T->split_k > 0) {
    S = T->split_k;
  } else {
    // Heuristic, measured on B300 over the sweep's shapes at M = 1 and 16
    // (slices x weight slots: 4096^2 8 x 4: 6.4 / 6.9 us; 11008 x 4096
    // 8 x 2 at M <= 8, 9.8 us, else 4 x 4, 12.0 us; 4096 x 11008 8 x 8 at
    // M <= 8, 11.6 us, else 8 x 4, 13.2 us): eight slices per n-tile, four
    // when there are more n-tiles than SMs half-way and two n8 token blocks
    S = (rows > 8 && 2 * ntl > sms) ? 4 : 8;
    while (S > ktl) S /= 2;
  }
  const bool s_ok = S >= 1 && S <= 16 && (S & (S - 1)) == 0 && S <= ktl;
  const int64_t nk_max = s_ok ? (ktl + S - 1) / S : 0;
  const int64_t ctas_per_sm = s_ok ? (ntl * S + sms - 1) / sms : 1;
  int ring = 4;
  if (T && T->kernel == 2 && T->stages) ring = T->stages;
  else if (rows <= 8 && ctas_per_sm > 2) ring = 2;      // many CTAs: small ones
  else if (rows <= 8 && nk_max > 4 && ctas_per_sm <= 2) ring = 8;   // long slices
  if (ring > nk_max) ring = (int)nk_max;
  if (ring < 1) ring = 1;
  const int mma_smem =
      s_ok ? mma_smem_bytes(packed_block_bytes(is_mx(L), st, has_zp), ring, (int)nk_max,
                            rows <= 8 ? 8 : 16, is_mx(L) ? 1 : 2, quant_in_lib(L))
           : 0;
  const bool mma_fits = s_ok && nk_max <= 64 && mma_smem <= device_max_smem();
  const bool mma_ok = !grouped && !is_w8(L) &&
                      L->gated_act == 0 && rows <= 16 && !(C && C->batch_invariant) &&
                      mma_fits;
  const int want = T ? T->kernel : 0;
  if (want == 2 && !mma_ok)
    return fail(QGEMM_ERR_UNSUPPORTED,
                "the small-M kernel takes dense INT4/UINT4/INT3/UINT3 GEMMs with scales in the "
                "activation dtype (or fp16 scales with bf16 activations), NVFP4 and W4A8-MXFP4 "
                "GEMMs, "
                "with m <= 16, not gated or "
                "batch-invariant, split_k a power of two <= 16 and <= k/128 and a slice that "
                "fits shared memory");
  P->kernel = 1;
  P->mma_splits = 0;
  // Heuristic: with no tuning field for the tcgen05 kernel set, the small-M
  // kernel takes every GEMM it can run (no tensor-memory set-up, no
  // split-tile finish through L2).
  const bool k1_tuned = T && (T->block_tok || T->stages || T->max_ctas || T->split_k);
  // NVFP4 weights cost about three integer operations per weight to decode,
  // which makes the small-M kernel issue-bound on large layers.  Measured on
  // B300 (bf16, us, small-M / tcgen05): 4096^2 8.4 / 9.5 at every M <= 16;
  // 11008 x 4096 13.1 / 14.1 at M <= 8, 18.8 / 14.3 at M = 16; 4096 x 11008
  // 14.7 / 14.5 at M = 1, 16.3 / 14.6 at M = 4.  So by default it takes them
  // up to 2^24 weights, or at M <= 8 with K <= 4096.
  const bool nv_small = !is_nv(L) || L->n * L->k <= (int64_t(1) << 24) ||
                        (rows <= 8 && L->k <= 4096);
  // 9-16 rows on a long K (at least twice as many k-tiles as n-tiles) go to
  // the tcgen05 kernel.  Measured on B300, UINT4 bf16 16 x 4096 x 11008: 12.3
  // us against 12.9-13.4 on the small-M kernel; at 8 rows, and at 16 rows on
  // 4096^2 and 11008 x 4096, the small-M kernel is faster.  W4A8 layers take
  // it above 8 rows at any shape (7168 x 2048, M = 16: 9.1 us with the
  // separate quantizer against 10.3 fused into the small-M kernel's two n8
  // token blocks; M = 8: 9.1 against 9.2).
  const bool long_k = rows > 8 && ktl >= 2 * ntl && !is_mx(L) && !is_nv(L) && !is_f16s(L);
  const bool mx_rows = rows > 8 && is_mx(L);
  const bool use_mma =
      want == 2 || (want == 0 && mma_ok && !k1_tuned && nv_small && !long_k && !mx_rows);
  if (use_mma) {
    if (ntl * S >= (int64_t(1) << 31)) return fail(QGEMM_ERR_UNSUPPORTED, "grid too large");
    P->kernel = 2;
    P->mma_splits = (int)S;
    P->mma_ring = ring;
    P->mma_nk_max = (int)nk_max;
    P->bt = 16;
    P->grid = (int)(ntl * S);
    P->split_cap = 0;
    P->st = st;
    P->off_s = kTileBytes;
    P->off_z = kTileBytes + packed_scale_bytes(is_mx(L), st);
    P->max_tiles = ntl;
    // the status word only: the slices meet in distributed shared memory (and
    // bf16 activations of a W4A8 layer are quantized inside the kernel)
    WorkspaceLayout w;
    w.counters_off = 256;
    w.counters_bytes = 0;
    w.partials_off = 256;
    w.partials_bytes = 0;
    w.total = 256;
    w.aq_off = w.aq_scale_off = 256;
    w.aq_bytes = 0;
    P->ws = w;
    return ok();
  }
  const int w_cap = (T && T->stages) ? T->stages : 16;
  if (w_cap < 2 || w_cap > 16) return fail(QGEMM_ERR_INVALID_ARG, "stages must be in [2, 16]");
  Geometry g;
  if (!make_geometry(bt, st, has_zp, is_mx(L), is_w8(L), E, w_cap, device_max_smem(), 0, &g))
    return fail(QGEMM_ERR_UNSUPPORTED, "tile does not fit shared memory");
  const int64_t kt = L->k / kTileK, nt = L->n / kTileN;
  int64_t tiles_bound;
  if (grouped)
    tiles_bound = ((rows + bt - 1) / bt + E) * nt;
  else
    tiles_bound = ((rows + bt - 1) / bt) * nt;
  if (tiles_bound >= (int64_t(1) << 31))
    return fail(QGEMM_ERR_UNSUPPORTED, "problem has more than 2^31 output tiles");
  // the device schedule works in 32-bit: stream-K units times CTAs < 2^31
  if (kt * (int64_t)sms * sms >= (int64_t(1) << 31))
    return fail(QGEMM_ERR_UNSUPPORTED, "k = %lld is too large for one GEMM", (long long)L->k);
  int grid = sms;
  if (T && T->max_ctas > 0 && T->max_ctas < grid) grid = T->max_ctas;
  if (!grouped) {
    const int64_t units = tiles_bound * kt;
    if (units < grid) grid = (int)(units > 0 ? units : 1);
    // Heuristic (16-bit MMA formats, neither a split cap nor a CTA cap
    // asked): whole tiles when the
    // k-tiles per CTA that stream-K saves over whole waves are worth less than
    // the fixed cost of its split tiles (the finishers' copy-in, add and store
    // at the end, the extra epilogue passes).  Measured on B300 per token tile
    // (BT 16 / 32 / 64 / 128): ~0.30 / 0.33 / 0.38 / 0.47 us per k-tile and
    // ~2.5 / 3 / 4.5 / 7 us of split cost: break-even at ~8 / 9 / 12 / 15.
    if (!is_mx(L) && cap == 0 && !(T && T->max_ctas > 0) && tiles_bound > 0) {
      const int64_t G = grid, Tt = tiles_bound;
      const double whole_units = (double)((Tt + G - 1) / G) * kt;
      int64_t W = Tt / G;
      if (W > 0 && Tt % G) --W;   // the two-wave stream-K of the device schedule
      const double sk_units = (double)W * kt + (double)(Tt - W * G) * kt / (double)G;
      const double breakeven = bt == 16 ? 8.0 : bt == 32 ? 9.0 : bt == 64 ? 12.0 : 15.0;
      if (whole_units - sk_units < breakeven) cap = 1;
    }
    // W4A8: whole tiles unless a tuning asks for splits (measured on B300,
    // N = 7168, K = 2048: M = 256 / 512 / 1024 15.9 / 24.0 / 36.3 us against
    // 24.3 / 28.9 / 39.7 with stream-K); they also keep no split-K state in
    // the workspace, where a layer on bf16 activations keeps its quantized rows
    if (is_mx(L) && cap == 0 && !(T && T->max_ctas > 0)) cap = 1;
    if (cap > 0 && tiles_bound * cap < grid)
      grid = (int)(tiles_bound > 0 ? tiles_bound * cap : 1);
  }
  if (grouped && quant_in_lib(L) && cap == 0 && !(T && T->max_ctas > 0)) cap = 1;
  // Cluster split: each tile's K range in S slices, one CTA each, the S CTAs
  // of a tile in one cluster summing their slices through distributed shared
  // memory (no workspace round trip, no wait on another tile's CTAs).
  // tuning.kernel = 3 asks for it (split_k = S, or 0 for the heuristic's);
  // otherwise the heuristic takes it for a dense GEMM when the tiles x S CTAs
  // fit the device at once and its estimate beats the persistent schedule's.
  const bool want_cl = T && T->kernel == 3;
  const bool cl_allowed = !grouped && !(C && C->batch_invariant) && bt <= 128 &&
                          !(T && T->max_ctas > 0) && tiles_bound > 0;
  if (want_cl && !cl_allowed)
    return fail(QGEMM_ERR_UNSUPPORTED,
                "the cluster split takes dense GEMMs with block_tok <= 128, not batch-invariant, "
                "without max_ctas");
  const int s_fixed = want_cl ? T->split_k : 0;
  if (want_cl && s_fixed != 0 && (s_fixed < 2 || s_fixed > 8 || s_fixed > kt))
    return fail(QGEMM_ERR_UNSUPPORTED, "a cluster split_k must be in [2, 8] and <= k/128");
  int cl = 0;
  Geometry gc;
  if (cl_allowed && (want_cl || !(T && T->split_k > 0))) {
    // a forced split with no count asked for takes at least two slices (in
    // several waves if the tiles need them)
    int S = s_fixed ? s_fixed
                    : (int)std::min<int64_t>(std::min<int64_t>(8, kt),
                                             std::max<int64_t>(want_cl ? 2 : 1,
                                                               sms / tiles_bound));
    for (; S >= 2; --S) {
      const int nu = (4 * (bt / 16) + S - 1) / S;   // 16-row chunks this CTA finishes
      if (!make_geometry(bt, st, has_zp, is_mx(L), is_w8(L), E, w_cap, device_max_smem(),
                         nu * (S - 1) * 2048, &gc)) {
        if (s_fixed) break;
        continue;
      }
      // a forced split may take several waves; the heuristic's must fit at once
      if (want_cl || tiles_bound <= w4a16_max_clusters(bt, fmt_of(L), S, gc.smem)) {
        cl = S;
        break;
      }
      if (s_fixed) break;
    }
    if (want_cl && cl == 0)
      return fail(QGEMM_ERR_UNSUPPORTED, "no cluster split of this tile fits shared memory");
    if (cl && !want_cl) {
      // Heuristic: per-CTA k-tiles at the measured per-k-tile cost (above),
      // plus the exchange, the rank-ordered sums and the stores (measured on
      // B300 at ~0.85 of stream-K's split cost: ~4 us at BT 64, ~6 us at BT
      // 128), against the persistent schedule's whole waves or stream-K.
      const double c = bt == 16 ? 0.30 : bt == 32 ? 0.33 : bt == 64 ? 0.38 : 0.47;
      const double split = bt == 16 ? 2.5 : bt == 32 ? 3.0 : bt == 64 ? 4.5 : 7.0;
      const int64_t G = grid, Tt = tiles_bound;
      const double whole = (double)((Tt + G - 1) / G) * kt * c;
      int64_t W = Tt / G;
      if (W > 0 && Tt % G) --W;
      const double sk = ((double)W * kt + (double)(Tt - W * G) * kt / (double)G) * c + split;
      const double t_sk = cap == 1 ? whole : std::min(whole, sk);
      const double t_cl = (double)((kt + cl - 1) / cl) * c + 0.85 * split;
      if (!(t_cl < t_sk)) cl = 0;
    }
    if (cl) {
      g = gc;
      cap = cl;
      grid = (int)(tiles_bound * cl);
    }
  }
  P->bt = bt;
  P->grid = grid;
  P->split_cap = cap;
  P->cluster = cl;
  P->st = st;
  P->off_s = packed_code_bytes(is_w8(L));                  // inside a packed block
  P->off_z = P->off_s + packed_scale_bytes(is_mx(L), st);
  P->g = g;
  P->max_tiles = tiles_bound;
  if (cl) {
    // the status word only: the slices meet in distributed shared memory
    WorkspaceLayout w;
    w.counters_off = w.partials_off = 256;
    w.counters_bytes = w.partials_bytes = 0;
    w.total = 256;
    w.aq_off = w.aq_scale_off = 256;
    w.aq_bytes = 0;
    P->ws = w;
  } else {
    P->ws = workspace_layout(tiles_bound, grid, bt);
  }
  if (quant_in_lib(L)) add_act_quant_region(&P->ws, rows, L->k);
  return ok();
}

// ------------------------------------------------------------ tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    const uint64_t dims[3], const uint64_t strides_bytes[2],
                    const uint32_t box[3], CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult res = fn(map, dtype, 3, const_cast<void*>(base), d, st, bx, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                    uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------ the W4A4 run

// Workspace: the status word, the K split's per-quadrant tile counters
// (cleared by each call's quantization kernel), its fp32 partial tiles, then
// the quantized activations (codes [rows, K/2], then e4m3 block scales
// [rows, K/16]).
struct W4A4Plan {
  int bt = 0;
  int splits = 1;
  int64_t grid = 0;
  size_t cnt_off = 0, part_off = 0, codes_off = 0, sb_off = 0, total = 0;
};

static qgemm_status w4a4_plan(const qgemm_layer_config* L, const qgemm_tuning_config* T,
                              int64_t rows, W4A4Plan* P) {
  *P = W4A4Plan();
  if (T && (T->stages || T->max_ctas || T->cta_pair || T->kernel > 1 || T->kernel < 0))
    return fail(QGEMM_ERR_UNSUPPORTED,
                "a W4A4 tuning may set block_tok, split_k (and kernel = 1) only");
  // Token tile: the tuning's; else the M range's, or above 16 rows the
  // smallest of 32 / 64 / 128 (up to the M range's) whose tiles still fit one
  // wave on the SMs, so that medium M keeps more SMs streaming.  Measured on
  // B300 (us, M range's tile / this): M = 64 4096^2 12.5 / 11.2 (32 tokens),
  // 4096 x 11008 20.4 / 17.4; M = 256 4096^2 16.0 / 13.4 (64), 4096 x 11008
  // 25.4 / 22.8; 11008 x 4096 keeps the M range's tile (86 feature tiles)
  int bt = rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
  if (T && T->block_tok) {
    bt = T->block_tok;
  } else if (rows > 16) {
    for (int b = 32; b < bt; b *= 2)
      if (((rows + b - 1) / b) * (L->n / kTileN) <= device_sm_count()) {
        bt = b;
        break;
      }
  }
  if (bt != 16 && bt != 32 && bt != 64 && bt != 128)
    return fail(QGEMM_ERR_UNSUPPORTED, "W4A4 block_tok %d not in {16, 32, 64, 128}", bt);
  const int64_t kt = L->k / kW4A4TileK;
  const int64_t tiles = ((rows + bt - 1) / bt) * (L->n / kTileN);
  // K slices per tile: the tuning's, else (few tiles of at most 64 tokens,
  // and 16-token tiles or K of at least 32 stages) as many as fill the SMs,
  // at least four stages each.  Measured on B300, us, whole tiles / split:
  // M = 1 4096^2 11.7 / 10.4 (4 slices); M = 1 / 16 / 64 4096 x 11008 19.6
  // / 20.1 / 22.3 against 13.9 / 14.6 / 20.6; M = 64 4096^2 14.4 / 17.8
  // and M = 256 (2 slices) 17.7 / 23.3: there the slices' partial round trip
  // costs more than the shorter K loop saves
  int64_t S = 1;
  if (T && T->split_k) {
    S = T->split_k;
    if (S < 1 || S > 64 || S > kt)
      return fail(QGEMM_ERR_UNSUPPORTED, "W4A4 split_k %d not in [1, min(64, k / 256)]",
                  T->split_k);
  } else if (tiles > 0 && tiles < device_sm_count() && bt <= 64 && (bt <= 16 || kt >= 32)) {
    S = std::min<int64_t>(std::min<int64_t>(16, kt / 4), device_sm_count() / tiles);
    if (S < 1) S = 1;
  }
  P->bt = bt;
  P->splits = (int)S;
  P->grid = tiles * S;
  if (P->grid >= (int64_t(1) << 31)) return fail(QGEMM_ERR_UNSUPPORTED, "grid too large");
  P->cnt_off = 256;
  P->part_off = P->cnt_off + (S > 1 ? (((size_t)tiles * 16 + 255) & ~size_t(255)) : 0);
  P->codes_off = P->part_off + (S > 1 ? (size_t)tiles * (size_t)S * (size_t)bt * 128 * 4 : 0);
  P->sb_off = P->codes_off + (((size_t)rows * (size_t)(L->k / 2) + 255) & ~size_t(255));
  P->total = P->sb_off + (((size_t)rows * (size_t)(L->k / 16) + 255) & ~size_t(255));
  return ok();
}

static qgemm_status run_w4a4(const qgemm_layer_config* L, const qgemm_tuning_config* T,
                             int64_t rows, const void* a, const float* a_scale, const void* w,
                             const void* bias, void* c, void* workspace, size_t ws_bytes,
                             cudaStream_t stream) {
  if (rows < 0 || rows > 0x7FFFFFFF) return fail(QGEMM_ERR_INVALID_ARG, "bad row count");
  if (rows == 0) return ok();
  if (!device_is_sm103()) return fail(QGEMM_ERR_UNSUPPORTED, "this library runs on sm_103 only");
  if (!a || !w || !c || (L->has_bias && !bias))
    return fail(QGEMM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!a_scale)
    return fail(QGEMM_ERR_INVALID_ARG, "W4A4 needs a_scale: the activations' fp32 tensor scale");
  if (!L->has_bias && bias) return fail(QGEMM_ERR_INVALID_ARG, "bias given with has_bias = 0");
  if (!aligned16(a) || !aligned16(w) || !aligned16(c) || (bias && !aligned16(bias)) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(a_scale) & 3u))
    return fail(QGEMM_ERR_INVALID_ARG, "pointers must be 16-byte aligned (a_scale 4-byte)");
  W4A4Plan P;
  qgemm_status st = w4a4_plan(L, T, rows, &P);
  if (st != QGEMM_OK) return st;
  if (!workspace || ws_bytes < P.total)
    return fail(QGEMM_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", P.total,
                ws_bytes);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  uint8_t* codes = wsb + P.codes_off;
  uint8_t* sb = wsb + P.sb_off;
  const uint64_t n = (uint64_t)L->n, k = (uint64_t)L->k;
  const uint8_t* wc = static_cast<const uint8_t*>(w);
  const uint8_t* wsc = wc + n * k / 2;
  CUtensorMap tm_w, tm_a, tm_ws, tm_as;
  if (!encode_tmap_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, wc, k / 2, n, k / 2, 128, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, k / 2, (uint64_t)rows, k / 2,
                      128, (uint32_t)P.bt, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tm_ws, CU_TENSOR_MAP_DATA_TYPE_UINT8, wsc, k / 16, n, k / 16, 16, 128,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tmap_2d(&tm_as, CU_TENSOR_MAP_DATA_TYPE_UINT8, sb, k / 16, (uint64_t)rows, k / 16,
                      16, (uint32_t)P.bt, CU_TENSOR_MAP_SWIZZLE_NONE))
    return fail(QGEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed for a W4A4 operand");
  W4A4Params p;
  memset(&p, 0, sizeof(p));
  p.m = (int)rows;
  p.n = (int)L->n;
  p.k = (int)L->k;
  p.kt = (int)(L->k / kW4A4TileK);
  p.nt = (int)(L->n / kTileN);
  p.mt = (int)((rows + P.bt - 1) / P.bt);
  p.a_ts = a_scale;
  p.w_ts = reinterpret_cast<const float*>(wsc + n * k / 16);
  p.bias = static_cast<const uint16_t*>(bias);
  p.c = static_cast<uint16_t*>(c);
  p.status = reinterpret_cast<int*>(wsb);
  p.wait_limit_ns = g_wait_limit_ns;
  p.splits = P.splits;
  p.cnt = reinterpret_cast<int*>(wsb + P.cnt_off);
  p.part = reinterpret_cast<float*>(wsb + P.part_off);
  p.part_rows = P.splits > 1 ? (long long)P.grid * P.bt : 0;   // tiles x slices x BT
  p.cnt_words = P.splits > 1 ? (int)(P.grid / P.splits * 4) : 0;
  // the quantization kernel also clears the K split's counters
  const int64_t n_cnt = P.splits > 1 ? P.grid / P.splits * 4 : 0;
  cudaError_t e = launch_act_quant_nvfp4(static_cast<const uint16_t*>(a), rows, (int64_t)k,
                                         a_scale, codes, sb, stream, p.cnt, (int)n_cnt);
  if (e != cudaSuccess) return cuda_fail(e, "NVFP4 activation quantization launch");
  e = launch_w4a4(tm_w, tm_a, tm_ws, tm_as, p, P.bt, stream);
  if (e != cudaSuccess) return cuda_fail(e, "W4A4 GEMM launch");
  return ok();
}

// ------------------------------------------------------------ the W4A16 run

static qgemm_status run_w4a16(const qgemm_layer_config* L, const qgemm_tuning_config* T,
                              const qgemm_compute_config* C, bool grouped, const int32_t* offsets,
                              int64_t rows, const void* a, const float* a_scale, const void* w,
                              const void* bias, void* c, void* workspace, size_t ws_bytes,
                              size_t clear_bytes, cudaStream_t stream) {
  if (rows < 0) return fail(QGEMM_ERR_INVALID_ARG, "row count is negative");
  if (rows > (1 << 30)) return fail(QGEMM_ERR_UNSUPPORTED, "row count above 2^30");
  if (rows == 0) return ok();
  if (!device_is_sm103()) return fail(QGEMM_ERR_UNSUPPORTED, "this library runs on sm_103 only");
  const bool has_zp = has_zeros(L);
  if (!a || !w || !c || (L->has_bias && !bias) || (grouped && !offsets))
    return fail(QGEMM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!L->has_bias && bias) return fail(QGEMM_ERR_INVALID_ARG, "bias given with has_bias = 0");
  const bool mx = is_mx(L);
  const bool qa = quant_in_lib(L);
  if (mx && !qa && !a_scale)
    return fail(QGEMM_ERR_INVALID_ARG, "the W4A8 path needs the per-row activation scales");
  if (qa && a_scale)
    return fail(QGEMM_ERR_INVALID_ARG,
                "a_scale must be NULL with bf16 activations (the library computes the scales)");
  if (!mx && a_scale) return fail(QGEMM_ERR_INVALID_ARG, "a_scale is only used by the W4A8 path");
  if (!aligned16(a) || !aligned16(w) || !aligned16(c) || (bias && !aligned16(bias)) ||
      !aligned16(workspace))
    return fail(QGEMM_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  Plan P;
  qgemm_status st = make_plan(L, T, C, rows, grouped, &P);
  if (st != QGEMM_OK) return st;
  if (!workspace || ws_bytes < P.ws.total)
    return fail(QGEMM_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", P.ws.total,
                ws_bytes);
  const bool fp16 = L->act_dtype == QGEMM_FP16;
  if (P.kernel == 2) {
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    W4A16MmaParams q;
    memset(&q, 0, sizeof(q));
    q.w = static_cast<const uint8_t*>(w);
    q.a = static_cast<const uint16_t*>(a);
    q.c = static_cast<uint16_t*>(c);
    q.bias = static_cast<const uint16_t*>(bias);
    q.status = reinterpret_cast<int*>(wsb);
    q.m = (int)rows;
    q.n = (int)L->n;
    q.k = (int)L->k;
    q.kt = (int)(L->k / kTileK);
    q.nt = (int)(L->n / kTileN);
    q.splits = P.mma_splits;
    q.ring = P.mma_ring;
    q.nk_max = P.mma_nk_max;
    q.wait_limit_ns = g_wait_limit_ns;
    q.block_bytes = packed_block_bytes(mx, P.st, has_zp);
    q.mx = mx ? 1 : 0;
    q.a_scale = a_scale;
    q.quant_act = qa ? 1 : 0;
    q.f16s = is_f16s(L) ? 1 : 0;
    q.nv = is_nv(L) ? 1 : 0;
    q.t_scales = is_nv(L) ? reinterpret_cast<const float*>(static_cast<const uint8_t*>(w) +
                                                           expert_packed_bytes(L))
                          : nullptr;
    q.s_off = P.off_s;
    q.z_off = P.off_z;
    q.sg_shift = L->group_size == 32 ? 0 : L->group_size == 64 ? 1 : 2;
    q.has_zp = has_zp ? 1 : 0;
    if (clear_bytes) {
      cudaError_t ce = cudaMemsetAsync(workspace, 0, clear_bytes, stream);
      if (ce != cudaSuccess) return cuda_fail(ce, "workspace clear");
    }
    // activations {128 bytes of k, rows, K / 128-byte chunks}: one box holds a
    // slice's k-tiles (16-bit: two chunks a k-tile; e4m3: one)
    CUtensorMap tmap_mma;
    const int eb = mx && !qa ? 1 : 2;
    const uint64_t rb = (uint64_t)L->k * eb;
    const uint64_t dims3[3] = {(uint64_t)(128 / eb), (uint64_t)rows, rb / 128};
    const uint64_t str3[2] = {rb, 128};
    const uint32_t box3[3] = {(uint32_t)(128 / eb), (uint32_t)(rows <= 8 ? 8 : 16),
                              (uint32_t)(eb * P.mma_nk_max)};
    if (!encode_tmap_3d(&tmap_mma,
                        eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                        : fp16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        a, dims3, str3, box3, CU_TENSOR_MAP_SWIZZLE_128B))
      return fail(QGEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed for the activation tensor");
    cudaError_t e = launch_w4a16_mma(tmap_mma, q, fp16, stream);
    if (e != cudaSuccess) return cuda_fail(e, "small-M GEMM launch");
    return ok();
  }
  // bf16 activations of a W4A8 layer: quantized per row into the workspace
  // (launched with the GEMM below, after every check), then run as e4m3 ones
  const void* a_bf16 = a;
  if (qa) {
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    a = wsb + P.ws.aq_off;
    a_scale = reinterpret_cast<const float*>(wsb + P.ws.aq_scale_off);
  }
  CUtensorMap tmap;
  // activation boxes [chunk][row][128 bytes]: the K axis split into 128-byte
  // chunks (64 16-bit or 128 e4m3 values) as the outermost box dimension, so
  // one box holds a stage's k-tiles in the 128-byte-swizzled operand layout
  const int r = units_per_stage(P.bt);
  const uint64_t row_bytes = (uint64_t)L->k * (mx ? 1 : 2);
  const uint64_t dims[3] = {(uint64_t)(mx ? 128 : 64), (uint64_t)rows, row_bytes / 128};
  const uint64_t strides[2] = {row_bytes, 128};
  const uint32_t box[3] = {(uint32_t)(mx ? 128 : 64), (uint32_t)P.bt,
                           (uint32_t)(mx ? r : 2 * r)};
  const bool tmap_ok = encode_tmap_3d(
      &tmap,
      mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8
         : fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
      a, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!tmap_ok)
    return fail(QGEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed for the activation tensor");
  const int E = L->num_experts;
  W4A16Params p;
  memset(&p, 0, sizeof(p));
  p.w = static_cast<const uint8_t*>(w);
  p.bias = static_cast<const uint16_t*>(bias);
  p.c = static_cast<uint16_t*>(c);
  p.a_scale = a_scale;
  p.rows = (int)rows;
  p.n = (int)L->n;
  p.k = (int)L->k;
  p.kt = (int)(L->k / kTileK);
  p.nt = (int)(L->n / kTileN);
  p.st = P.st;
  p.group = L->group_size;
  p.sg_shift = L->group_size == 32 ? 0 : L->group_size == 64 ? 1 : 2;
  p.has_zp = has_zp ? 1 : 0;
  p.gated = L->gated_act != 0;
  p.split_cap = P.split_cap;
  p.expert_offsets = offsets;
  p.num_experts = E;
  p.w_expert_stride = (long long)expert_packed_bytes(L);
  p.t_scales = is_nv(L) ? reinterpret_cast<const float*>(static_cast<const uint8_t*>(w) +
                                                         (size_t)E * expert_packed_bytes(L))
                        : nullptr;
  p.block_bytes = packed_block_bytes(mx, P.st, has_zp, is_w8(L));
  p.s_off = P.off_s;
  p.z_off = P.off_z;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.status = reinterpret_cast<int*>(ws);
  p.counters = reinterpret_cast<int*>(ws + P.ws.counters_off);
  p.partials = reinterpret_cast<float*>(ws + P.ws.partials_off);
  p.deterministic = C->deterministic ? 1 : 0;
  p.max_tiles = P.max_tiles;
  p.x_stages = P.g.x_stages;
  p.x_bytes = P.g.x_bytes;
  p.w_stages = P.g.w_stages;
  p.w_bytes = P.g.w_bytes;
  p.rw = P.g.rw;
  p.off_w = P.g.off_w;
  p.off_epi = P.g.off_epi;
  p.off_bar = P.g.off_bar;
  p.off_recv = P.g.off_recv;
  p.cluster = P.cluster;
  p.smem_bytes = P.g.smem;
  // several token tiles per weight block: keep weights in L2 rather than
  // marking them first to evict
  p.w_reuse = grouped ? (rows > (int64_t)E * P.bt) : (rows > P.bt);
  // the dense schedule's constants and divisors (the device re-derives the
  // grouped one from the expert offsets)
  {
    const int64_t T = grouped ? 0 : ((rows + P.bt - 1) / P.bt) * (L->n / kTileN);
    const int64_t G = P.grid;
    int64_t W = T / G;
    // uncapped: one whole wave fewer when tiles are left over, so that every
    // CTA's stream-K range spans at least a tile and each split tile has two
    // contributors, the later of which meets it as its first item
    if (P.split_cap == 0 && W > 0 && T % G) --W;
    const int64_t U = (T - W * G) * p.kt;
    p.sk_t = (int)T;
    p.sk_w = (int)W;
    p.sk_u = (int)U;
    // the r remaining tiles' units go to min(G, U) CTAs; with a cap, each
    // tile to exactly min(cap, G / r) CTAs (tile-aligned; 1: whole tiles)
    int64_t gs = U < G ? U : G;
    if (P.split_cap > 0 && U > 0) {
      const int64_t r = U / p.kt;
      const int64_t per = P.split_cap < G / r ? P.split_cap : G / r;
      if (r * per < gs) gs = r * per;
    }
    p.sk_gs = (int)gs;
    p.div_kt = make_fastdiv((uint32_t)p.kt);
    p.div_nt = make_fastdiv((uint32_t)p.nt);
    p.div_gs = make_fastdiv(p.sk_gs > 0 ? (uint32_t)p.sk_gs : 1u);
    p.div_u = make_fastdiv(p.sk_u > 0 ? (uint32_t)p.sk_u : 1u);
  }
  // a split tile's finisher copies the other contributors' fp32 sum (BT x 128)
  // into the activation ring when it is large enough
  p.fix_smem = (int64_t)P.g.x_stages * P.g.x_bytes >= (int64_t)P.bt * kTileN * 4;
  // the last item's per-chunk staging: BT * 512 bytes of sums, then 4 warps x
  // BT/16 chunks x 2 KB
  p.last_stage = (int64_t)P.g.x_stages * P.g.x_bytes >= (int64_t)P.bt * 1024;
  p.wait_limit_ns = g_wait_limit_ns;
  // output [rows, n] of 16-bit values, written by 16-row x 32-column tensor
  // stores; a gated output [rows, n/2] by 16-row x 16-column ones
  CUtensorMap tmap_c;
  const uint64_t n_out = p.gated ? (uint64_t)L->n / 2 : (uint64_t)L->n;
  if (!encode_tmap_2d(&tmap_c, CU_TENSOR_MAP_DATA_TYPE_UINT16, c, n_out, (uint64_t)rows,
                      n_out * 2, p.gated ? 16 : 32, 16, CU_TENSOR_MAP_SWIZZLE_NONE))
    return fail(QGEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed for the output tensor");
  const int fmt = fmt_of(L);
  if (clear_bytes) {
    cudaError_t ce = cudaMemsetAsync(workspace, 0, clear_bytes, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "workspace clear");
  }
  if (qa && P.split_cap != 1 && P.cluster == 0) {
    // a split-K plan asked for by a tuning on a layer whose quantized rows share
    // the workspace: another plan's rows may lie where this plan keeps its
    // counters and accumulators, so they start cleared
    cudaError_t ce = cudaMemsetAsync(static_cast<uint8_t*>(workspace) + P.ws.counters_off, 0,
                                     P.ws.partials_off + P.ws.partials_bytes - P.ws.counters_off,
                                     stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "workspace clear");
  }
  if (qa) {   // the GEMM waits on this grid before it reads the codes and scales
    cudaError_t qe = launch_act_quant_fp8(
        static_cast<const uint16_t*>(a_bf16), rows, L->k,
        static_cast<uint8_t*>(const_cast<void*>(a)), const_cast<float*>(a_scale), stream);
    if (qe != cudaSuccess) return cuda_fail(qe, "activation quantization launch");
  }
  cudaError_t e = launch_w4a16(tmap, tmap_c, p, P.bt, fmt, grouped, P.grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "W4A16 GEMM launch");
  return ok();
}

int run_dense_clearing(const void* layer, const void* compute, const void* tuning, int64_t m,
                       const void* a, const float* a_scale, const void* packed, const void* bias,
                       void* c, void* workspace, size_t ws_bytes, size_t clear_bytes,
                       cudaStream_t stream) {
  const qgemm_layer_config* L = static_cast<const qgemm_layer_config*>(layer);
  const qgemm_compute_config* C = static_cast<const qgemm_compute_config*>(compute);
  qgemm_status st = check_layer(L);
  if (st != QGEMM_OK) return st;
  st = check_compute(C, L, false);
  if (st != QGEMM_OK) return st;
  if (is_w4a4(L)) {
    if (clear_bytes && workspace) {
      cudaError_t ce = cudaMemsetAsync(workspace, 0, clear_bytes, stream);
      if (ce != cudaSuccess) return cuda_fail(ce, "workspace clear");
    }
    return run_w4a4(L, static_cast<const qgemm_tuning_config*>(tuning), m, a, a_scale, packed,
                    bias, c, workspace, ws_bytes, stream);
  }
  return run_w4a16(L, static_cast<const qgemm_tuning_config*>(tuning), C, false, nullptr, m, a,
                   a_scale, packed, bias, c, workspace, ws_bytes, clear_bytes, stream);
}

int set_last_error(int status, const char* message) {
  g_last_error = message;
  return status;
}

int dense_workspace_bytes(const void* layer, const void* compute, const void* tuning, int64_t m,
                          size_t* must_clear, size_t* total) {
  const qgemm_layer_config* L = static_cast<const qgemm_layer_config*>(layer);
  qgemm_status st = check_layer(L);
  if (st != QGEMM_OK) return st;
  if (is_w4a4(L)) {   // only the status word starts at zero (the call clears its counters)
    W4A4Plan W;
    st = w4a4_plan(L, static_cast<const qgemm_tuning_config*>(tuning), m > 0 ? m : 1, &W);
    if (st != QGEMM_OK) return st;
    *must_clear = 256;
    *total = W.total;
    return QGEMM_OK;
  }
  Plan P;
  st = make_plan(L, static_cast<const qgemm_tuning_config*>(tuning),
                 static_cast<const qgemm_compute_config*>(compute), m > 0 ? m : 1, false, &P);
  if (st != QGEMM_OK) return st;
  // the status word and tile counters start at zero, and so do the split-K
  // accumulators of the atomic reduction (the quantized activations, last,
  // are written in full before they are read)
  *must_clear = P.ws.total - P.ws.aq_bytes;
  *total = P.ws.total;
  return QGEMM_OK;
}

}  // namespace qg

using namespace qg;

extern "C" {

qgemm_status qgemm_packed_size(const qgemm_layer_config* layer, size_t* bytes) {
  qgemm_status st = check_layer(layer);
  if (st != QGEMM_OK) return st;
  if (!bytes) return fail(QGEMM_ERR_INVALID_ARG, "bytes is NULL");
  if (is_w4a4(layer)) {   // codes [N, K/2], block scales [N, K/16], the tensor scale
    *bytes = (size_t)layer->n * (size_t)layer->k / 2 + (size_t)layer->n * (size_t)layer->k / 16 + 16;
    return ok();
  }
  *bytes = (size_t)layer->num_experts * expert_packed_bytes(layer);
  if (is_nv(layer)) *bytes += (size_t)((layer->num_experts + 3) / 4) * 16;   // tensor scales
  return ok();
}

qgemm_status qgemm_pack_weights(const qgemm_layer_config* layer, const void* qweight,
                                const void* scales, const void* qzeros, void* packed,
                                void* stream) {
  qgemm_status st = check_layer(layer);
  if (st != QGEMM_OK) return st;
  const bool has_zp = has_zeros(layer);
  const bool nv = is_nv(layer);   // qzeros carries the fp32 tensor scales
  if (!qweight || !scales || !packed || ((has_zp || nv) && !qzeros))
    return fail(QGEMM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!has_zp && !nv && qzeros)
    return fail(QGEMM_ERR_INVALID_ARG, "zero points given for a format without");
  if (!aligned16(packed) || !aligned16(qweight))
    return fail(QGEMM_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  cudaError_t e;
  if (is_w4a4(layer)) {
    // W4A4 reads the standard format as it is: the copy lays codes, block
    // scales and the tensor scale end to end
    if ((reinterpret_cast<uintptr_t>(qzeros) & 3u) != 0)
      return fail(QGEMM_ERR_INVALID_ARG, "NVFP4 tensor scales must be 4-byte aligned");
    const size_t cb = (size_t)layer->n * (size_t)layer->k / 2;
    const size_t sbb = (size_t)layer->n * (size_t)layer->k / 16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* dst = static_cast<uint8_t*>(packed);
    e = cudaMemcpyAsync(dst, qweight, cb, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst + cb, scales, sbb, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst + cb + sbb, qzeros, sizeof(float), cudaMemcpyDefault, s);
  } else if (nv) {
    if ((reinterpret_cast<uintptr_t>(qzeros) & 3u) != 0)
      return fail(QGEMM_ERR_INVALID_ARG, "NVFP4 tensor scales must be 4-byte aligned");
    e = launch_repack_nvfp4(static_cast<const uint8_t*>(qweight),
                            static_cast<const uint8_t*>(scales), static_cast<const float*>(qzeros),
                            static_cast<uint8_t*>(packed), layer->n, layer->k,
                            layer->num_experts, layer->act_dtype == QGEMM_FP16,
                            layer->gated_act != 0, static_cast<cudaStream_t>(stream));
  } else if (is_mx(layer)) {
    if ((reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
      return fail(QGEMM_ERR_INVALID_ARG, "MXFP4 scales must be 4-byte aligned");
    e = launch_repack_mxfp4(static_cast<const uint8_t*>(qweight),
                            static_cast<const uint8_t*>(scales), static_cast<uint8_t*>(packed),
                            layer->n, layer->k, layer->num_experts, layer->gated_act != 0,
                            static_cast<cudaStream_t>(stream));
  } else if (is_w8(layer)) {
    e = launch_repack_w8(static_cast<const int32_t*>(qweight),
                         static_cast<const uint16_t*>(scales), static_cast<const int32_t*>(qzeros),
                         static_cast<uint8_t*>(packed), layer->n, layer->k, layer->group_size,
                         layer->weight_format == QGEMM_W_INT8_SYM ? 1 : 0, layer->num_experts,
                         layer->gated_act != 0, static_cast<cudaStream_t>(stream));
  } else {
    e = launch_repack_w4(static_cast<const int32_t*>(qweight),
                         static_cast<const uint16_t*>(scales), static_cast<const int32_t*>(qzeros),
                         static_cast<uint8_t*>(packed), layer->n, layer->k, layer->group_size,
                         (layer->weight_format == QGEMM_W_INT4_SYM ||
                          layer->weight_format == QGEMM_W_INT3_SYM)
                             ? 1
                             : 0,
                         layer->num_experts, layer->gated_act != 0, is_w3(layer) ? 3 : 4,
                         static_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return cuda_fail(e, "repack launch");
  return ok();
}

qgemm_status qgemm_workspace_size(const qgemm_layer_config* layer,
                                  const qgemm_compute_config* compute,
                                  const qgemm_tuning_config* tuning, int64_t m, size_t* bytes) {
  if (!bytes) return fail(QGEMM_ERR_INVALID_ARG, "bytes is NULL");
  qgemm_status st = check_layer(layer);
  if (st != QGEMM_OK) return st;
  const bool grouped = compute && compute->gemm_type == QGEMM_GEMM_GROUPED;
  st = check_compute(compute, layer, grouped);
  if (st != QGEMM_OK) return st;
  if (m < 0) return fail(QGEMM_ERR_INVALID_ARG, "m is negative");
  if (is_w4a4(layer)) {
    if (grouped) return fail(QGEMM_ERR_UNSUPPORTED, "W4A4 runs dense GEMMs");
    W4A4Plan W;
    st = w4a4_plan(layer, tuning, m > 0 ? m : 1, &W);
    if (st != QGEMM_OK) return st;
    *bytes = W.total;
    return ok();
  }
  Plan P;
  st = make_plan(layer, tuning, compute, m > 0 ? m : 1, grouped, &P);
  if (st != QGEMM_OK) return st;
  *bytes = P.ws.total;
  return ok();
}

qgemm_status qgemm_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (!workspace || bytes == 0) return fail(QGEMM_ERR_INVALID_ARG, "empty workspace");
  cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "workspace memset");
  return ok();
}

qgemm_status qgemm_run(const qgemm_layer_config* layer, const qgemm_compute_config* compute,
                       const qgemm_tuning_config* tuning, int64_t m, const void* a,
                       const float* a_scale, const void* packed, const void* bias, void* c,
                       void* workspace, size_t workspace_bytes, void* stream) {
  qgemm_status st = check_layer(layer);
  if (st != QGEMM_OK) return st;
  st = check_compute(compute, layer, false);
  if (st != QGEMM_OK) return st;
  if (is_w4a4(layer))
    return run_w4a4(layer, tuning, m, a, a_scale, packed, bias, c, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream));
  return run_w4a16(layer, tuning, compute, false, nullptr, m, a, a_scale,
                   packed, bias, c, workspace,
                   workspace_bytes, 0, static_cast<cudaStream_t>(stream));
}

qgemm_status qgemm_grouped_run(const qgemm_layer_config* layer,
                               const qgemm_compute_config* compute,
                               const qgemm_tuning_config* tuning, const int32_t* expert_offsets,
                               int64_t total_rows, const void* a, const float* a_scale,
                               const void* packed, const void* bias, void* c, void* workspace,
                               size_t workspace_bytes, void* stream) {
  qgemm_status st = check_layer(layer);
  if (st != QGEMM_OK) return st;
  st = check_compute(compute, layer, true);
  if (st != QGEMM_OK) return st;
  if (is_w4a4(layer)) return fail(QGEMM_ERR_UNSUPPORTED, "W4A4 runs dense GEMMs");
  return run_w4a16(layer, tuning, compute, true, expert_offsets,
                   total_rows, a, a_scale, packed, bias, c,
                   workspace, workspace_bytes, 0, static_cast<cudaStream_t>(stream));
}

qgemm_status qgemm_quantize_act_fp8(const void* x, int64_t m, int64_t k, void* a8,
                                    float* a_scale, void* stream) {
  if (m < 0 || k <= 0) return fail(QGEMM_ERR_INVALID_ARG, "bad shape");
  if (k % 8) return fail(QGEMM_ERR_UNSUPPORTED, "k must be a multiple of 8");
  if (m > (1 << 30) || k > (1 << 30)) return fail(QGEMM_ERR_UNSUPPORTED, "m or k above 2^30");
  if (m == 0) return ok();
  if (!x || !a8 || !a_scale) return fail(QGEMM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(a8) & 7u) ||
      (reinterpret_cast<uintptr_t>(a_scale) & 3u))
    return fail(QGEMM_ERR_INVALID_ARG, "x must be 16-byte, a8 8-byte, a_scale 4-byte aligned");
  cudaError_t e = launch_act_quant_fp8(static_cast<const uint16_t*>(x), m, k,
                                       static_cast<uint8_t*>(a8), a_scale,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "activation quantization launch");
  return ok();
}

qgemm_status qgemm_quantize_act_nvfp4(const void* x, int64_t m, int64_t k, const float* a_ts,
                                      void* codes, void* block_scales, void* stream) {
  if (m < 0 || k <= 0) return fail(QGEMM_ERR_INVALID_ARG, "bad shape");
  if (k % 16) return fail(QGEMM_ERR_UNSUPPORTED, "k must be a multiple of 16");
  if (m > (1 << 30) || k > (1 << 30)) return fail(QGEMM_ERR_UNSUPPORTED, "m or k above 2^30");
  if (m == 0) return ok();
  if (!x || !a_ts || !codes || !block_scales)
    return fail(QGEMM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(codes) & 7u) ||
      (reinterpret_cast<uintptr_t>(a_ts) & 3u))
    return fail(QGEMM_ERR_INVALID_ARG, "x must be 16-byte, codes 8-byte, a_ts 4-byte aligned");
  cudaError_t e = launch_act_quant_nvfp4(static_cast<const uint16_t*>(x), m, k, a_ts,
                                         static_cast<uint8_t*>(codes),
                                         static_cast<uint8_t*>(block_scales),
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "NVFP4 activation quantization launch");
  return ok();
}

qgemm_status qgemm_moe_permute(const int32_t* topk_ids, int64_t t, int32_t topk, int32_t e,
                               int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                               const void* a, void* a_perm, int64_t hidden, void* stream) {
  if (t < 0 || topk <= 0 || e <= 0 || hidden <= 0)
    return fail(QGEMM_ERR_INVALID_ARG, "bad shape");
  if (e > kMaxPermuteExperts)
    return fail(QGEMM_ERR_UNSUPPORTED, "at most %d experts", kMaxPermuteExperts);
  if (hidden % 8) return fail(QGEMM_ERR_UNSUPPORTED, "hidden must be a multiple of 8");
  if (t * topk > (1 << 28)) return fail(QGEMM_ERR_UNSUPPORTED, "too many slots");
  if (!offsets || (t > 0 && (!topk_ids || !perm || !inv_perm || !a || !a_perm)))
    return fail(QGEMM_ERR_INVALID_ARG, "a required pointer is NULL");
  if ((a && !aligned16(a)) || (a_perm && !aligned16(a_perm)))
    return fail(QGEMM_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  cudaError_t err = launch_moe_permute(topk_ids, t, topk, e, offsets, perm, inv_perm,
                                       static_cast<const uint16_t*>(a),
                                       static_cast<uint16_t*>(a_perm), hidden,
                                       static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "MoE permute launch");
  return ok();
}

qgemm_status qgemm_moe_silu_mul(const void* gu, int64_t rows, int64_t inter, void* h,
                                void* stream) {
  if (rows < 0 || inter <= 0 || inter % 8) return fail(QGEMM_ERR_INVALID_ARG, "bad shape");
  if (rows == 0) return ok();
  if (!gu || !h || !aligned16(gu) || !aligned16(h))
    return fail(QGEMM_ERR_INVALID_ARG, "pointers must be non-NULL and 16-byte aligned");
  cudaError_t err = launch_silu_mul(static_cast<const uint16_t*>(gu), rows, inter,
                                    static_cast<uint16_t*>(h), static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "SiLU launch");
  return ok();
}

qgemm_status qgemm_moe_combine(const void* y2, const int32_t* inv_perm,
                               const float* topk_weights, int64_t t, int32_t topk,
                               int64_t hidden, void* y, void* stream) {
  if (t < 0 || topk <= 0 || hidden <= 0 || hidden % 8)
    return fail(QGEMM_ERR_INVALID_ARG, "bad shape");
  if (t == 0) return ok();
  if (!y2 || !inv_perm || !topk_weights || !y || !aligned16(y2) || !aligned16(y))
    return fail(QGEMM_ERR_INVALID_ARG, "pointers must be non-NULL and 16-byte aligned");
  cudaError_t err = launch_combine(static_cast<const uint16_t*>(y2), inv_perm, topk_weights, t,
                                   topk, hidden, static_cast<uint16_t*>(y),
                                   static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "combine launch");
  return ok();
}

qgemm_status qgemm_debug_dequant(const qgemm_layer_config* layer, const void* packed,
                                 void* out_kn, void* stream) {
  qgemm_status st = check_layer(layer);
  if (st != QGEMM_OK) return st;
  if (!packed || !out_kn) return fail(QGEMM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (is_w4a4(layer))
    return fail(QGEMM_ERR_UNSUPPORTED, "a W4A4 buffer holds the standard tensors as they are");
  cudaError_t e;
  if (is_mx(layer))
    e = launch_debug_mx_codes(static_cast<const uint8_t*>(packed), static_cast<uint8_t*>(out_kn),
                              layer->n, layer->k, layer->gated_act != 0,
                              static_cast<cudaStream_t>(stream));
  else
    e = launch_debug_dequant(static_cast<const uint8_t*>(packed), static_cast<uint16_t*>(out_kn),
                             layer->n, layer->k, layer->group_size,
                             has_zeros(layer) ? 1 : 0,
                             layer->act_dtype == QGEMM_FP16, is_nv(layer), is_f16s(layer),
                             is_w8(layer),
                             layer->gated_act != 0, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "debug dequant launch");
  return ok();
}

qgemm_status qgemm_check_status(void* workspace, void* stream) {
  if (!workspace) return fail(QGEMM_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int word = 0;
  e = cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (word != 0) {
    const int zero = 0;
    e = cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    if (word & kStatusTimeout)
      return fail(QGEMM_ERR_TIMEOUT, "a kernel gave up a bounded wait (status 0x%x)", word);
    if (word & kStatusCheck)
      return fail(QGEMM_ERR_DEVICE, "an index check of the checked build failed (status 0x%x)",
                  word);
    return fail(QGEMM_ERR_DEVICE, "a kernel reported inconsistent inputs (status %d)", word);
  }
  return ok();
}

void qgemm_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns = ns; }

int qgemm_checked_build(void) { return kChecked ? 1 : 0; }

qgemm_status qgemm_checked_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  const int word = checked_word_read_and_clear();
  if (word < 0) return fail(QGEMM_ERR_CUDA, "check word read");
  if (word & kStatusCheck)
    return fail(QGEMM_ERR_DEVICE, "an index check of the checked build failed (status 0x%x)",
                word);
  return ok();
}

qgemm_status qgemm_checked_selftest(void* workspace, void* stream) {
  if (!kChecked) return fail(QGEMM_ERR_UNSUPPORTED, "this is not the checked build");
  if (!workspace || !aligned16(workspace))
    return fail(QGEMM_ERR_INVALID_ARG, "workspace must be a 16-byte aligned device pointer");
  cudaError_t e = launch_check_selftest(static_cast<int*>(workspace),
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return ok();
}

qgemm_status qgemm_describe_plan(const qgemm_layer_config* layer,
                                 const qgemm_compute_config* compute, int64_t m, char* buf,
                                 size_t len) {
  std::string rec;
  qgemm_status st = check_layer(layer);
  const bool grouped = compute && compute->gemm_type == QGEMM_GEMM_GROUPED;
  if (st == QGEMM_OK) st = check_compute(compute, layer, grouped);
  W4A4Plan W;
  if (st == QGEMM_OK && is_w4a4(layer))
    st = grouped ? fail(QGEMM_ERR_UNSUPPORTED, "W4A4 runs dense GEMMs")
                 : w4a4_plan(layer, nullptr, m > 0 ? m : 1, &W);
  if (st != QGEMM_OK) {
    rec = std::string("rejected: ") + g_last_error;
  } else if (is_w4a4(layer)) {
    char tmp[384], split[48];
    if (W.splits > 1)
      snprintf(split, sizeof(split), "k_slices_%d_last_arrival_sum", W.splits);
    else
      snprintf(split, sizeof(split), "whole_tiles");
    const int sms = device_sm_count();
    snprintf(tmp, sizeof(tmp),
             "kernel=w4a4_tcgen05_mxf4nvf4 weights=nvfp4 group=16 scales=e4m3 act=nvfp4 out=bf16 "
             "n=%lld k=%lld m=%lld experts=1 block_tok=%d stages=6 items=%lld grid=%lld smem=%d "
             "workspace=%zu epilogue=%s split=%s act_quant=separate_kernel "
             "device=sm_103",
             (long long)layer->n, (long long)layer->k, (long long)m, W.bt, (long long)W.grid,
             (long long)(sms > 0 && W.grid > sms ? sms : W.grid), w4a4_smem_bytes(W.bt), W.total,
             layer->has_bias ? "bias" : "plain", split);
    rec = tmp;
  } else {
    Plan P;
    st = make_plan(layer, nullptr, compute, m > 0 ? m : 1, grouped, &P);
    if (st != QGEMM_OK) {
      rec = std::string("rejected: ") + g_last_error;
    } else {
      static const char* wf[] = {"int4_sym", "uint4_zp", "mxfp4",    "nvfp4",
                                 "int8_sym", "uint8_zp", "int3_sym", "uint3_zp"};
      static const char* dt[] = {"fp16", "bf16", "fp8e4m3", "nvfp4"};
      static const char* sf[] = {"fp16", "bf16", "e8m0", "e4m3"};
      char tmp[512];
      snprintf(tmp, sizeof(tmp),
               "kernel=%s%s weights=%s group=%d scales=%s act=%s out=%s n=%lld k=%lld "
               "m=%lld experts=%d block_tok=%d act_slots=%d weight_slots=%dx%d grid=%d smem=%d "
               "workspace=%zu epilogue=%s split=%s act_quant=%s "
               "device=sm_103",
               P.kernel == 2 ? "w4a16_mma_sync_smallm"
               : is_mx(layer) ? "w4a8_tcgen05_mxf8f6f4_swapab" : "w4a16_tcgen05_swapab",
               grouped ? "_grouped" : "", wf[layer->weight_format], layer->group_size,
               sf[layer->scale_format], dt[layer->act_dtype], dt[layer->out_dtype], (long long)layer->n,
               (long long)layer->k, (long long)m, layer->num_experts, P.bt, P.g.x_stages,
               P.g.w_stages, P.g.rw, P.grid, P.g.smem, P.ws.total,
               layer->gated_act ? "silu_glu" : "plain",
               P.kernel == 2     ? "k_slices"
               : P.cluster > 1   ? (P.cluster == 2   ? "cluster_k2"
                                    : P.cluster == 3 ? "cluster_k3"
                                    : P.cluster == 4 ? "cluster_k4"
                                    : P.cluster == 5 ? "cluster_k5"
                                    : P.cluster == 6 ? "cluster_k6"
                                    : P.cluster == 7 ? "cluster_k7"
                                                     : "cluster_k8")
               : P.split_cap == 1 ? "whole_tiles"
                                  : "stream_k",
               !quant_in_lib(layer) ? "none" : P.kernel == 2 ? "fused" : "separate_kernel");
      rec = tmp;
    }
  }
  if (buf && len) {
    strncpy(buf, rec.c_str(), len - 1);
    buf[len - 1] = 0;
  }
  return st;
}

const char* qgemm_status_string(qgemm_status s) {
  switch (s) {
    case QGEMM_OK: return "QGEMM_OK";
    case QGEMM_ERR_INVALID_ARG: return "QGEMM_ERR_INVALID_ARG";
    case QGEMM_ERR_UNSUPPORTED: return "QGEMM_ERR_UNSUPPORTED";
    case QGEMM_ERR_WORKSPACE: return "QGEMM_ERR_WORKSPACE";
    case QGEMM_ERR_CUDA: return "QGEMM_ERR_CUDA";
    case QGEMM_ERR_TIMEOUT: return "QGEMM_ERR_TIMEOUT";
    case QGEMM_ERR_DEVICE: return "QGEMM_ERR_DEVICE";
    default: return "QGEMM_UNKNOWN_STATUS";
  }
}

const char* qgemm_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
