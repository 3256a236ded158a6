// K3: expert histogram, prefix scan and token permutation — the grouping step of the grouped GEMM
// ("Strata" 3090 tuning, xdnf.cn/news/329730, §3.2: tokens routed to the same expert are gathered
// into one small matrix group, and all groups go through one grouped-GEMM launch).
//
// One CTA of 1024 threads performs a stable counting sort of the T*k routed rows by expert id, so
// row order is (expert, token) and the result is deterministic:
//   pass 1  each warp owns a contiguous range of the flattened [T, k] id array and counts it into its
//           own histogram row (__match_any_sync groups equal ids inside a 32-row step);
//   scan    counts[e] = sum over warps; offsets = exclusive scan; each warp's histogram row becomes
//           the first output position of its rows of expert e;
//   pass 2  the same walk assigns positions: base + rank among equal ids in the step.
// The CTA then lists the active segments (shared expert first, then routed experts with rows, in
// id order) and the per-segment work-item counts that the grouped GEMM walks.
#include "kernels.cuh"

namespace strata {

// Exclusive scan over the 1024 threads of the block; returns the exclusive prefix, writes the total.
__device__ int block_exclusive_scan(int v, int* scratch /* [32] */, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
    int winc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += n;
    }
    scratch[lane] = winc - w;  // exclusive prefix of warp totals
    if (lane == 31) scratch[32] = winc;
  }
  __syncthreads();
  const int res = scratch[warp] + inc - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(1024) permute_kernel(PermuteArgs a) {
  extern __shared__ int hist[];  // [32][E]
  __shared__ int scratch[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E;
  const int R = a.T * a.k;
  for (int i = tid; i < 32 * E; i += 1024) hist[i] = 0;
  __syncthreads();

  const int per_warp = (R + 31) / 32;
  const int rbeg = min(R, warp * per_warp), rend = min(R, rbeg + per_warp);
  const unsigned lt_mask = (1u << lane) - 1u;
  // pass 1: per-warp histograms
  for (int base = rbeg; base < rend; base += 32) {
    const int r = base + lane;
    const unsigned active = __ballot_sync(0xffffffffu, r < rend);
    if (r < rend) {
      int e = a.ids[r];
      if (e < 0 || e >= E) {
        set_status(a.status, STRATA_DEV_BAD_ID);
        e = -1;
      }
      const unsigned m = __match_any_sync(active, e);
      if (e >= 0 && (m & lt_mask) == 0) hist[warp * E + e] += __popc(m);
      __syncwarp(active);
    }
  }
  __syncthreads();
  // counts and offsets (E <= 1024: one expert per thread)
  int cnt = 0;
  if (tid < E)
    for (int w = 0; w < 32; ++w) cnt += hist[w * E + tid];
  int total;
  const int off = block_exclusive_scan(tid < E ? cnt : 0, scratch, &total);
  if (tid < E) {
    a.counts[tid] = cnt;
    a.offsets[tid] = off;
    int run = off;
    for (int w = 0; w < 32; ++w) {
      const int c = hist[w * E + tid];
      hist[w * E + tid] = run;
      run += c;
    }
  }
  if (tid == 0) a.offsets[E] = total;
  __syncthreads();
  // pass 2: positions
  for (int base = rbeg; base < rend; base += 32) {
    const int r = base + lane;
    const unsigned active = __ballot_sync(0xffffffffu, r < rend);
    if (r < rend) {
      int e = a.ids[r];
      if (e < 0 || e >= E) e = -1;
      const unsigned m = __match_any_sync(active, e);
      if (e >= 0) {
        const int pos = hist[warp * E + e] + __popc(m & lt_mask);
        a.perm[pos] = r / a.k;
        a.inv[r] = pos;
      }
      __syncwarp(active);
      if (e >= 0 && (m & lt_mask) == 0) hist[warp * E + e] += __popc(m);
      __syncwarp(active);
    }
  }
  // the shared expert's rows: identity order after the routed rows
  if (a.has_shared)
    for (int t = tid; t < a.T; t += 1024) a.perm[R + t] = t;

  if (a.seg_expert == nullptr) return;
  // active segments: shared first (largest), then routed experts in id order
  const int sh = (a.has_shared && a.T > 0) ? 1 : 0;
  const int flag = (tid < E && cnt > 0) ? 1 : 0;
  int nseg_routed;
  const int sidx = block_exclusive_scan(flag, scratch, &nseg_routed) + sh;
  const int nseg = nseg_routed + sh;
  if (flag) {
    a.seg_expert[sidx] = tid;
    a.seg_row0[sidx] = a.offsets[tid];  // written above by this thread
    a.seg_rows[sidx] = cnt;
  }
  if (sh && tid == 0) {
    a.seg_expert[0] = E;
    a.seg_row0[0] = R;
    a.seg_rows[0] = a.T;
  }
  __syncthreads();
  // work items per segment, prefix over segments (segment s is handled by thread s)
  int my_rows = 0;
  if (tid < nseg) my_rows = a.seg_rows[tid];
  const int chunks = (my_rows + a.tokc - 1) / a.tokc;
  int tot_gu, tot_dn;
  const int pre_gu = block_exclusive_scan(tid < nseg ? chunks * a.mtiles_gu : 0, scratch, &tot_gu);
  const int pre_dn = block_exclusive_scan(tid < nseg ? chunks * a.mtiles_dn : 0, scratch, &tot_dn);
  if (tid < nseg) {
    a.seg_item_gu[tid] = pre_gu;
    a.seg_item_dn[tid] = pre_dn;
  }
  if (tid == 0) {
    a.seg_item_gu[nseg] = tot_gu;
    a.seg_item_dn[nseg] = tot_dn;
    a.hdr->nseg = nseg;
    a.hdr->n_items_gu = tot_gu;
    a.hdr->n_items_dn = tot_dn;
  }
}

cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(32) * a.E * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  permute_kernel<<<1, 1024, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace strata
