// Self-test of the bounded device waits, outside any data path: the mbarrier wait of the TMA-fed
// grouped GEMMs (tc::mbar_wait) and the counter spin of the fused router (spin_until_geq) are run
// on a barrier and a counter that nothing completes. Each must give up after its limit, flag
// STRATA_DEV_TIMEOUT and return, leaving the context usable.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace strata {

// words: [0] status word, [1] a counter nothing increments (zero), [2] / [3] set to 1 when the
// mbarrier wait / the counter spin gave up.
__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint32_t* words,
                                                                   long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  tc::mbar_init(&bar, 1);
  abort_flag = 0;
  tc::fence_barrier_init();
  // phase 0 of `bar` completes on one arrival, and none is ever made
  const bool a = tc::mbar_wait(&bar, 0u, &abort_flag, words, limit);
  const bool b = spin_until_geq(words + 1, 1u, limit, words);
  words[2] = a ? 0u : 1u;
  words[3] = b ? 0u : 1u;
}

cudaError_t launch_wait_selftest(uint32_t* words, long long limit, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(words, limit);
  return cudaGetLastError();
}

}  // namespace strata
