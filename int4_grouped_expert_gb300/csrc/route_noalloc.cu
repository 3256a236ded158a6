// strata_route_topk_noalloc: the router + top-k + grouping of strata_route_topk for callers that
// may not allocate device memory at call time and cannot hand the library a workspace of their
// own — for example plugin interfaces whose enqueue step must not allocate, code that runs while
// a CUDA graph is being captured (cudaMalloc is not allowed then), or processes whose device
// memory is owned up front by one custom allocator.
//
// The scratch lives in a fixed array in the library's device globals instead of a caller
// workspace. Every GPU that loads the library holds this array until the process exits. Host code
// cannot use the array's name as a device address, so the first call on each device looks the
// address up with cudaGetSymbolAddress (with that device current) and keeps it.
#include <mutex>

#include "kernels.cuh"

namespace {

// Holds the router's partial logits and the status header; requests that need more return
// STRATA_ERR_UNSUPPORTED.
__device__ __align__(256) unsigned char g_route_scratch[STRATA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device (looked up once per device).
strata_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return STRATA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return STRATA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
      return STRATA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return STRATA_OK;
}

}  // namespace

extern "C" strata_status strata_route_topk_noalloc(const void* x_bf16, const float* w_router,
                                                   const float* bias, int64_t T, int64_t H,
                                                   int32_t E, int32_t k, uint32_t flags,
                                                   int32_t* ids, float* gates, int32_t* counts,
                                                   int32_t* offsets, int32_t* perm, int32_t* inv,
                                                   strata_stream stream) {
  if (T < 0 || E < 1 || k < 1) return STRATA_ERR_INVALID_ARG;
  const size_t need = strata_route_workspace_size(T, E, k);
  if (need == 0) return STRATA_ERR_INVALID_ARG;
  if (need > STRATA_NOALLOC_SCRATCH_BYTES) return STRATA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const strata_status s = scratch_on_current_device(&scratch);
  if (s != STRATA_OK) return s;
  // strata_route_topk clears the scratch header (status word) on the stream before its kernels.
  return strata_route_topk(x_bf16, w_router, bias, T, H, E, k, flags, ids, gates, counts, offsets,
                           perm, inv, scratch, STRATA_NOALLOC_SCRATCH_BYTES, stream);
}
