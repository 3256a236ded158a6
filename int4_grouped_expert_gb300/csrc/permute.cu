// K3: expert histogram, prefix scan and token permutation for large batches — one CTA of 1024
// threads runs the stable counting sort of group_rows.cuh over all T*k routed rows. (Small decode
// batches do the same work in the last CTA of the fused router, router.cu.)
#include "group_rows.cuh"

namespace strata {

__global__ void __launch_bounds__(1024) permute_kernel(PermuteArgs a) {
  extern __shared__ int gsm[];
  group_rows<32>(a, a.ids, carve_group_smem(gsm, 32, a.E));
}

cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t stream) {
  const size_t smem = group_smem_ints(32, a.E) * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  permute_kernel<<<1, 1024, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace strata
