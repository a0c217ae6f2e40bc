// Attention-core backward that allocates nothing: for callers that may not
// allocate device memory at the point of the call, such as a framework's
// allocator running its own out-of-memory or defragmentation path, or a
// runtime whose device memory budget is reserved up front and fully claimed.
// The scratch of the backward (the per-tile LSE/Delta records and, when a
// chunk holds fewer query heads than a KV group, the fp32 dK/dV carry) lives
// in a fixed array in this module's static device memory instead of a
// caller-supplied workspace.
#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "upipe.h"
#include "upipe_internal.h"

namespace {

// Every device that loads this library holds this array until the process
// exits.  All calls share it, and it keeps the previous call's contents.
__device__ __align__(256) unsigned char g_upipe_noalloc_scratch[UPIPE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::atomic<void*> g_scratch_addr[kMaxDev];  // device address of the array, per device
std::mutex g_scratch_mu;

}  // namespace

extern "C" int upipe_attn_core_bwd_noalloc(const upipe_cfg* cfg, const uint16_t* q, const uint16_t* k,
                                           const uint16_t* v, const uint16_t* o, const float* lse,
                                           const uint16_t* dout_o, uint16_t* dq, uint16_t* dk, uint16_t* dv,
                                           void* stream) {
  const size_t need = upipe_workspace_bytes(cfg, 1, 1, 0);
  if (need == 0) return UPIPE_ERR_INVALID_ARG;
  if (need > UPIPE_NOALLOC_SCRATCH_BYTES) return UPIPE_ERR_SCRATCH_LIMIT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UPIPE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDev) return UPIPE_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return UPIPE_ERR_CUDA;
  if (major != 10 || minor != 3) return UPIPE_ERR_UNSUPPORTED_DEVICE;
  void* scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!scratch) {
    // Once per device, with that device current: the array's name is only a
    // host-side stand-in; kernels need its device address.
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    scratch = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!scratch) {
      if (cudaGetSymbolAddress(&scratch, g_upipe_noalloc_scratch) != cudaSuccess || scratch == nullptr)
        return UPIPE_ERR_CUDA;
      g_scratch_addr[dev].store(scratch, std::memory_order_release);
    }
  }
  // Nothing in the scratch has to start at zero: every record and carry is
  // written before it is read within one call.  Profiling events are not
  // recorded for this call's launches (recording may create events).
  upipe::ProfilingOff no_events;
  return upipe_attn_core_bwd(cfg, q, k, v, o, lse, dout_o, dq, dk, dv, scratch, UPIPE_NOALLOC_SCRATCH_BYTES,
                             stream);
}
