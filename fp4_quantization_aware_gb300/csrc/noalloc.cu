// attnqat_bwd_noalloc: the backward for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain a workspace: code that runs where a
// device allocation is not allowed or not possible (a host callback, a runtime
// that forbids cudaMalloc after start-up, an embedding with its own fixed
// memory budget and no allocator hook). This entry point gives them the
// backward with its scratch space (Q^, K^, V^ and their NVFP4 encodings,
// delta, the FP32 dQ accumulator, the split-tile counters and dK/dV slots) in
// a statically sized device array that the library declares itself, so the
// call allocates nothing.
//
// Limits and sharing:
//  - The array holds kNoAllocScratchBytes (32 MiB). A problem whose
//    attnqat_bwd_workspace_bytes() exceeds it is rejected with
//    ATTNQAT_ERR_WORKSPACE before anything is enqueued.
//  - Every GPU that loads this module holds the array until the process exits.
//  - All calls on a device share the one array and it keeps the last call's
//    contents. The parts that must start at zero (the FP32 dQ accumulator, the
//    split-tile counters and the FP32 dK/dV slots of split tiles) are all
//    cleared by the preprocess step of every call. Calls whose executions
//    overlap on the GPU (different streams, or different host threads without
//    ordering between them) race on the array and give wrong results.
//  - The first call on each device looks up the array's device address with
//    cudaGetSymbolAddress (with that device current). Under CUDA's lazy module
//    loading (the default since CUDA 12.2) this lookup is what loads the
//    module and reserves the 32 MiB, so the first call can fail with
//    ATTNQAT_ERR_CUDA on a full device: make it at start-up, before any stream
//    capture and before a memory budget applies.
//  - The address is cached per device index for the life of the CUDA context;
//    a device reset (cudaDeviceReset) between calls would leave it stale.
#include <mutex>

#include "../../include/attnqat.h"
#include "kernels.h"

namespace attnqat {
void set_error_message(const char* msg);
}

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// In host code this name is only a stand-in for the device array: its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" attnqat_status attnqat_bwd_noalloc(const attnqat_problem* p, const void* dout, const void* q,
                                              const void* k, const void* v, const void* o_hp, const float* lse,
                                              void* dq, void* dk, void* dv, void* stream) {
  const size_t need = attnqat_bwd_workspace_bytes(p);
  if (need == 0) return attnqat_check_support(p);   // reports why the problem is not supported
  if (need > kNoAllocScratchBytes) {
    attnqat::set_error_message(
        "attnqat_bwd_noalloc: the problem needs more scratch than the 32 MiB static array holds; "
        "use attnqat_bwd with a caller workspace");
    return ATTNQAT_ERR_WORKSPACE;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    attnqat::set_error_message("attnqat_bwd_noalloc: no usable current device");
    return ATTNQAT_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || ptr == nullptr) {
        attnqat::set_error_message("attnqat_bwd_noalloc: cudaGetSymbolAddress of the static scratch failed");
        return ATTNQAT_ERR_CUDA;
      }
      g_scratch_ptr[dev] = ptr;
    }
    scratch = g_scratch_ptr[dev];
  }
  return attnqat_bwd(p, dout, q, k, v, o_hp, lse, dq, dk, dv, scratch, kNoAllocScratchBytes, stream);
}
