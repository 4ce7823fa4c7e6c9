// qgemm_run_noalloc: the dense GEMM of qgemm_run without a caller workspace.
//
// Some callers cannot allocate device memory at the moment they run a GEMM:
// code that executes under a memory-pool or allocator lock it does not own,
// plugins loaded into a host program that manages every device byte itself,
// or start-up and recovery paths that must not touch the allocator at all.
// They can still pass their own inputs and outputs, but not the split-K
// scratch.  For them this entry point takes the scratch from a fixed array
// that lives inside the library image: it allocates nothing and calls no
// allocating routine.
//
// The array is kNoAllocScratchBytes (32 MiB) per GPU, held until the process
// exits.  The CUDA runtime may load the library's device code lazily, so the
// array becomes resident on a device when the first call made with that
// device current looks up its address; that lookup can fail for lack of
// device memory, in which case the call returns QGEMM_ERR_CUDA and the next
// call tries again.  Make that first call early, before any CUDA stream
// capture.  All calls share the one array and it keeps what the last call
// left in it: calls that can overlap on the GPU (different streams, or
// different host threads) race on it and must be serialised by the caller.
// Each call, once its arguments have passed every check, zeroes the part of
// the array its launch needs (status word, split-K tile counters and split-K
// accumulators; cudaMemsetAsync on its stream, which allocates nothing) just
// before the launch; a rejected call queues nothing.  A problem whose scratch
// exceeds the array is rejected with QGEMM_ERR_UNSUPPORTED.

#include <cstdio>
#include <mutex>

#include "../../include/qgemm.h"
#include "internal.h"

namespace qg {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
bool g_scratch_ok[kMaxDevices];
std::mutex g_scratch_mu[kMaxDevices];

// Device address of the scratch array on the current device.  The name of a
// __device__ array in host code is only a host-side stand-in, so the address
// comes from the runtime, with that device current.  Only a successful
// lookup is kept; a failed one (say the module could not be loaded for lack
// of memory) is retried by the next call.
cudaError_t scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu[dev]);
  if (!g_scratch_ok[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();   // do not leave the error for the caller's next CUDA call
      return e;
    }
    g_scratch_ptr[dev] = p;
    g_scratch_ok[dev] = true;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace qg

extern "C" qgemm_status qgemm_run_noalloc(const qgemm_layer_config* layer,
                                          const qgemm_compute_config* compute,
                                          const qgemm_tuning_config* tuning, int64_t m,
                                          const void* a, const float* a_scale,
                                          const void* packed, const void* bias, void* c,
                                          void* stream) {
  using namespace qg;
  if (!compute || compute->gemm_type != QGEMM_GEMM_DENSE)
    return qgemm_status(set_last_error(QGEMM_ERR_INVALID_ARG,
                                       "qgemm_run_noalloc runs dense GEMMs only"));
  if (m < 0) return qgemm_status(set_last_error(QGEMM_ERR_INVALID_ARG, "m is negative"));
  if (m == 0)
    return qgemm_run(layer, compute, tuning, 0, a, a_scale, packed, bias, c, nullptr, 0, stream);
  size_t must_clear = 0, need = 0;
  const int st = dense_workspace_bytes(layer, compute, tuning, m, &must_clear, &need);
  if (st != QGEMM_OK) return qgemm_status(st);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "qgemm_run_noalloc: this problem needs %zu bytes of split-K scratch, the static "
             "scratch holds %zu; use qgemm_run with a caller workspace",
             need, kNoAllocScratchBytes);
    return qgemm_status(set_last_error(QGEMM_ERR_UNSUPPORTED, msg));
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess)
    return qgemm_status(set_last_error(QGEMM_ERR_CUDA, cudaGetErrorString(e)));
  // the remaining checks run before the clear, so a rejected call queues nothing
  return qgemm_status(run_dense_clearing(layer, compute, tuning, m, a, a_scale, packed, bias, c,
                                         scratch, kNoAllocScratchBytes, must_clear,
                                         static_cast<cudaStream_t>(stream)));
}

extern "C" qgemm_status qgemm_noalloc_check_status(void* stream) {
  using namespace qg;
  void* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess)
    return qgemm_status(set_last_error(QGEMM_ERR_CUDA, cudaGetErrorString(e)));
  return qgemm_check_status(scratch, stream);
}
