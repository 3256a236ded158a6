// strata_route_topk_noalloc: the router + top-k + grouping of strata_route_topk for callers that
// may not allocate device memory at call time and cannot hand the library a workspace of their
// own — for example plugin interfaces whose enqueue step must not allocate, code that runs while
// a CUDA graph is being captured (cudaMalloc is not allowed then), or processes whose device
// memory is owned up front by one custom allocator.
//
// The scratch lives in a fixed array in the library's device globals instead of a caller
// workspace. Every GPU that loads the library holds this array until the process exits. Host code
// cannot use the array's name as a device address, so each call made outside stream capture looks
// the address up with cudaGetSymbolAddress (with the device current) and keeps it for calls made
// while a stream captures.
#include <mutex>

#include "kernels.cuh"

namespace {

// Holds the router's partial logits and the status header; requests that need more return
// STRATA_ERR_UNSUPPORTED.
__device__ __align__(256) unsigned char g_route_scratch[STRATA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_route_scratch in the current context. The lookup is repeated on every call
// made outside stream capture, so a reset device or another context gets its own module's
// address; during a capture the address kept from the last uncaptured call on the device is used
// (no lookup runs while the stream captures).
strata_status scratch_on_current_device(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return STRATA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return STRATA_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return STRATA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap == cudaStreamCaptureStatusNone || !g_scratch_ptr[dev]) {
    if (cap != cudaStreamCaptureStatusNone) return STRATA_ERR_UNSUPPORTED;  // no earlier call
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
  // the same argument checks, in the same order, as strata_route_topk; then the size limit
  const strata_status chk = strata::check_route_args(x_bf16, w_router, T, H, E, k, flags, ids,
                                                     gates, counts, offsets, perm, inv);
  if (chk != STRATA_OK) return chk;
  const size_t need = strata_route_workspace_size(T, E, k);
  if (need == 0) return STRATA_ERR_INVALID_ARG;
  if (need > STRATA_NOALLOC_SCRATCH_BYTES) return STRATA_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  const strata_status s = scratch_on_current_device(st, &scratch);
  if (s != STRATA_OK) return s;
  // strata_route_topk clears the scratch header (status word) on the stream before its kernels.
  return strata_route_topk(x_bf16, w_router, bias, T, H, E, k, flags, ids, gates, counts, offsets,
                           perm, inv, scratch, STRATA_NOALLOC_SCRATCH_BYTES, stream);
}
