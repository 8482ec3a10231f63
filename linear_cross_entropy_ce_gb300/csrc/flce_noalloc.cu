// flce_fwd_bwd_noalloc: the fused linear cross-entropy forward+backward for
// callers that cannot allocate device memory themselves -- for example code
// running inside a CUDA graph capture or a custom allocator hook, plugins
// whose host framework owns every cudaMalloc, or environments where
// allocating would break a memory budget fixed in advance.  Its scratch is a
// file-scope static device array of FLCE_NOALLOC_WORKSPACE_BYTES, created
// when the library's device code is loaded on a GPU and held by that GPU
// until the process exits.  The caller still passes inputs and outputs.
#include <mutex>

#include "flce.h"
#include "flce_internal.h"

namespace flce {
flce_status fwd_bwd_on_workspace(const void* hidden, const void* weight, const int32_t* targets, int64_t N,
                                 int64_t H, int64_t V, int32_t ignore_index, uint32_t flags, float* loss,
                                 int32_t* n_valid, float* row_loss, void* grad_hidden, float* grad_weight,
                                 void* workspace, size_t workspace_bytes, void* stream);
}

namespace {

// Shared by every call on a device; it keeps the last call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FLCE_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current.
flce_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FLCE_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return FLCE_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return FLCE_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FLCE_OK;
}

}  // namespace

extern "C" flce_status flce_fwd_bwd_noalloc(const void* hidden, const void* weight, const int32_t* targets,
                                            int64_t N, int64_t H, int64_t V, int32_t ignore_index,
                                            uint32_t flags, float* loss, int32_t* n_valid, float* row_loss,
                                            void* grad_hidden, float* grad_weight, void* stream) {
  void* ws = nullptr;
  const flce_status s = scratch_for_current_device(&ws);
  if (s != FLCE_OK) return s;
  // The plan is the largest token chunk that fits in the static array;
  // sizes whose smallest plan does not fit are rejected with FLCE_EWORKSPACE.
  return flce::fwd_bwd_on_workspace(hidden, weight, targets, N, H, V, ignore_index, flags, loss, n_valid,
                                    row_loss, grad_hidden, grad_weight, ws, FLCE_NOALLOC_WORKSPACE_BYTES, stream);
}
