// K5: weighted un-permute / combine of the expert outputs. Each token's output is the sum of its k
// routed expert outputs weighted by their gates, plus the always-on shared expert with gate 1
// ("GLM-5.3-Flash on one 4090", haowenji.com/articles/x-2109226022155796480, §01: 8 routed + 1
// shared expert per token), summed in fp32 in a fixed order (j = 0..k-1, shared, residual) and
// rounded once to bf16.
#include "kernels.cuh"

namespace strata {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y,
                                                      const float* __restrict__ gates,
                                                      const int* __restrict__ inv,
                                                      const __nv_bfloat16* __restrict__ x, int T,
                                                      int H, int k, int has_shared, int R,
                                                      int residual, __nv_bfloat16* __restrict__ out,
                                                      const int* __restrict__ T_dev) {
  // The token's routing (gates, rows) comes from the router, which completed before the GEMMs
  // that precede this grid started, and x is the layer input: both are read before waiting for
  // the down GEMM, so only the y rows are on the path after it.
  __shared__ float s_gate[STRATA_MAX_TOPK];
  __shared__ int s_row[STRATA_MAX_TOPK];
  const int t = blockIdx.x;
  if (T_dev) {  // a padded batch: only its live tokens have rows (routed rows first, then shared)
    const int live = live_tokens(T_dev, T);
    if (t >= live) return;
    R = live * k;
  }
  if (threadIdx.x < k) {
    const int64_t tk = static_cast<int64_t>(t) * k + threadIdx.x;
    s_gate[threadIdx.x] = gates[tk];
    s_row[threadIdx.x] = inv[tk];
  }
  const int64_t H4 = H / 4;
  const int64_t c0 = blockIdx.y * blockDim.x + threadIdx.x;
  uint2 xres = make_uint2(0u, 0u);
  if (residual && c0 < H4) xres = reinterpret_cast<const uint2*>(x + static_cast<int64_t>(t) * H)[c0];
  __syncthreads();
  griddep_wait();  // y comes from the down GEMM
  for (int64_t c = c0; c < H4; c += gridDim.y * blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const float g = s_gate[j];
      const int row = s_row[j];
      // a row outside the routed rows (the grouping skipped a bad expert id, or a timed-out
      // top-k left the buffer unwritten; both set a device status bit) contributes nothing
      if (row < 0 || row >= R) continue;
      const float4 v = __ldcg(reinterpret_cast<const float4*>(y + static_cast<int64_t>(row) * H) + c);
      acc.x = fmaf(g, v.x, acc.x); acc.y = fmaf(g, v.y, acc.y);
      acc.z = fmaf(g, v.z, acc.z); acc.w = fmaf(g, v.w, acc.w);
    }
    if (has_shared) {
      const float4 v = reinterpret_cast<const float4*>(y + static_cast<int64_t>(R + t) * H)[c];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (residual) {
      const uint2 raw = c == c0 ? xres : reinterpret_cast<const uint2*>(x + static_cast<int64_t>(t) * H)[c];
      const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&raw);
      const float2 a = __bfloat1622float2(p[0]), b = __bfloat1622float2(p[1]);
      acc.x += a.x; acc.y += a.y; acc.z += b.x; acc.w += b.y;
    }
    uint2 o;
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(out + static_cast<int64_t>(t) * H)[c] = o;
  }
}

cudaError_t launch_combine(const float* y, const float* gates, const int* inv, const void* x,
                           int64_t T, int64_t H, int k, int has_shared, int64_t R, int residual,
                           void* out, const int* T_dev, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  // one float4 of one token per thread: T x ceil(H / 1024) CTAs
  dim3 grid(static_cast<unsigned>(T), static_cast<unsigned>((H / 4 + 255) / 256));
  return launch_kernel(combine_kernel, grid, dim3(256), 0, stream, true, y, gates, inv,
                       static_cast<const __nv_bfloat16*>(x), static_cast<int>(T),
                       static_cast<int>(H), k, has_shared, static_cast<int>(R), residual,
                       static_cast<__nv_bfloat16*>(out), T_dev);
}

}  // namespace strata
