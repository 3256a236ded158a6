// K2: router logits + softmax + top-k ("Strata" MoE tuning notes, lpnh.cn/news/2730718, §2.3,
// point 1: softmax and top-k selection fused into one kernel; routing engine of the 102.7 tok/s
// write-up, zwxr.cn/news/276292, §3.2: softmax over the logits, partial sort, expert ids out).
//
// Decode batches (T <= 64): ONE launch, route_small_kernel. Each CTA owns 1-8 router rows (about
// one CTA per SM); the 8 warps split each row along H, dot their slice with every token and the
// slices are summed in shared memory in a fixed order. The last CTA to finish (a device-scope
// counter) runs softmax and top-k for every token and then groups the routed rows
// (group_rows.cuh).
//
// Large batches: router_logits_tc_kernel (tensor cores, exact three-way bf16 split of the fp32
// router, compensated accumulation), router_topk_kernel (one warp per token), then the permute
// kernel.
//
// Top-k order: descending logit, ties to the lower expert id; gates = softmax probabilities of the
// chosen experts (fp32, expf), renormalised over the k only with STRATA_RENORM.
#include "group_rows.cuh"

namespace strata {

// ----------------------------------------------------------------------------- shared pieces

// Order-preserving map of a float to uint32 (larger float -> larger key; -0 folded into +0).
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Best key of one lane's NPL keys and its slot, by a pairwise tree (ties keep the lower slot, which
// is the lower expert id).
// Slots whose bit is set in `taken` count as empty (a bit mask, not stores into key[]: an indexed
// store would move the array to local memory).
template <int N>
__device__ __forceinline__ void lane_best(const uint32_t (&key)[N], uint32_t taken, uint32_t& bk,
                                          int& bi) {
  uint32_t k2[N];
  int i2[N];
#pragma unroll
  for (int i = 0; i < N; ++i) { k2[i] = ((taken >> i) & 1u) ? 0u : key[i]; i2[i] = i; }
#pragma unroll
  for (int w = 1; w < N; w <<= 1) {
#pragma unroll
    for (int i = 0; i + w < N; i += 2 * w)
      if (k2[i + w] > k2[i]) { k2[i] = k2[i + w]; i2[i] = i2[i + w]; }
  }
  bk = k2[0];
  bi = i2[0];
}

// Softmax + top-k of TPW tokens at once by one warp (their dependency chains interleave). Token j
// is row t0 + j * tstride of lg (row stride ld) and is skipped if that is >= T; E <= 32 * NPL.
// Lane l keeps the order-preserving keys of experts e = l + 32 i in registers with its best
// remaining one. Each of the k rounds takes the warp-wide largest best key with one redux.sync and
// the lowest expert id among the lanes holding it with a second; that lane marks the slot taken
// and every lane re-takes its best. The rounds are branch-free, so the TPW chains interleave. Gates are computed by lanes 0..k-1 at the end.
// kGlobal: lg is global memory written by other CTAs of this grid (read through L2).
template <int NPL, int TPW, bool kGlobal>
__device__ __forceinline__ void warp_topk_multi(const float* lg, int64_t ld, int t0, int tstride,
                                                int T, int E, int k, uint32_t flags, int* ids,
                                                float* gates) {
  const int lane = threadIdx.x & 31;
  uint32_t key[TPW][NPL];
  // all loads first, unconditional (clamped address), so that they are in flight together
  float v[TPW][NPL];
#pragma unroll
  for (int j = 0; j < TPW; ++j) {
    const int t = t0 + j * tstride;
    const float* row = lg + static_cast<int64_t>(t < T ? t : 0) * ld;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      const float* src = row + (e < E ? e : E - 1);
      v[j][i] = kGlobal ? __ldcg(src) : *src;
    }
  }
#pragma unroll
  for (int j = 0; j < TPW; ++j) {
    const bool tok = t0 + j * tstride < T;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      key[j][i] = (tok && lane + 32 * i < E) ? float_key(v[j][i]) : 0u;
  }
  uint32_t bk[TPW], taken[TPW];
  int bi[TPW];
  float mx[TPW], sum[TPW];
#pragma unroll
  for (int j = 0; j < TPW; ++j) {
    taken[j] = 0u;
    lane_best<NPL>(key[j], 0u, bk[j], bi[j]);
    mx[j] = key_float(__reduce_max_sync(0xffffffffu, bk[j]));
  }
#pragma unroll
  for (int j = 0; j < TPW; ++j) {
    float sj = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (lane + 32 * i < E) sj += expf(key_float(key[j][i]) - mx[j]);
    sum[j] = sj;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int j = 0; j < TPW; ++j) sum[j] += __shfl_xor_sync(0xffffffffu, sum[j], o);
  }
  uint32_t my_key[TPW], my_id[TPW];
#pragma unroll
  for (int j = 0; j < TPW; ++j) { my_key[j] = 0u; my_id[j] = 0u; }
#pragma unroll 1
  for (int r = 0; r < k; ++r) {
    // one phase at a time over the TPW tokens: the warp-wide reductions are kept in program
    // order, so interleaving them by hand is what lets the tokens' latencies overlap
    uint32_t m[TPW], cand[TPW], eb[TPW];
#pragma unroll
    for (int j = 0; j < TPW; ++j) m[j] = __reduce_max_sync(0xffffffffu, bk[j]);
#pragma unroll
    for (int j = 0; j < TPW; ++j) {
      cand[j] = static_cast<uint32_t>(lane + 32 * bi[j]);
      eb[j] = __reduce_min_sync(0xffffffffu, bk[j] == m[j] ? cand[j] : 0xFFFFFFFFu);
    }
#pragma unroll
    for (int j = 0; j < TPW; ++j) {
      if (lane == r) { my_key[j] = m[j]; my_id[j] = eb[j]; }
      if (cand[j] == eb[j] && bk[j] == m[j]) taken[j] |= 1u << bi[j];
      lane_best<NPL>(key[j], taken[j], bk[j], bi[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < TPW; ++j) {
    const int t = t0 + j * tstride;
    const float g = lane < k ? expf(key_float(my_key[j]) - mx[j]) / sum[j] : 0.f;
    float gsum = g;
    if (flags & STRATA_RENORM) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
    }
    if (t < T && lane < k) {
      ids[static_cast<int64_t>(t) * k + lane] = static_cast<int>(my_id[j]);
      gates[static_cast<int64_t>(t) * k + lane] = (flags & STRATA_RENORM) ? g / gsum : g;
    }
  }
}

template <int TPW, bool kGlobal>
__device__ void warp_softmax_topk(const float* lg, int64_t ld, int t0, int tstride, int T, int E,
                                  int k, uint32_t flags, int* ids, float* gates) {
  const int npl = (E + 31) / 32;
#define STRATA_TOPK_CASE(N) \
  warp_topk_multi<N, TPW, kGlobal>(lg, ld, t0, tstride, T, E, k, flags, ids, gates)
  if (npl <= 1) STRATA_TOPK_CASE(1);
  else if (npl <= 2) STRATA_TOPK_CASE(2);
  else if (npl <= 4) STRATA_TOPK_CASE(4);
  else if (npl <= 8) STRATA_TOPK_CASE(8);
  else if (npl <= 10) STRATA_TOPK_CASE(10);
  else if (npl <= 16 || TPW > 2) STRATA_TOPK_CASE(16);  // callers keep E <= 512 for TPW > 2
  else STRATA_TOPK_CASE(32);
#undef STRATA_TOPK_CASE
}

// ----------------------------------------------------------------------------- decode: fused

constexpr int kRsWarps = 8;
constexpr long long kRouterWaitCycles = 2000000000ll;  // bound of the top-k CTAs' wait

int route_small_epc(int E, int num_sms) {
  int epc = 1;  // experts per CTA: about one CTA per SM
  while (epc < 8 && (E + epc - 1) / epc > num_sms) epc *= 2;
  return epc;
}

// dynamic shared memory of the last CTA (bytes): the grouping scratch, then ids and gates [T*k]
__host__ __device__ static bool route_small_compact_group(const RouteSmallArgs& a) {
  return a.grp.chunk_list != nullptr && a.T * a.k <= kGroupSmallMaxR;
}
__host__ __device__ static size_t route_small_ids_off(const RouteSmallArgs& a) {
  const size_t g = route_small_compact_group(a) ? group_small_ints(kRsWarps, a.E, a.T * a.k)
                                                : group_smem_ints(kRsWarps, a.E);
  return (g * 4 + 15) & ~static_cast<size_t>(15);
}
__host__ __device__ static size_t route_small_smem(const RouteSmallArgs& a) {
  return route_small_ids_off(a) + static_cast<size_t>(a.T) * a.k * 8;
}

template <bool kF16>
__global__ void __launch_bounds__(256) route_small_kernel(RouteSmallArgs a) {
  extern __shared__ __align__(16) unsigned char rs_smem[];
  __shared__ float red[kRsWarps][kRouteSmallMaxT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a.T sizes the launch and the shared memory; with a device token count (a fixed-size batch
  // with padding) the live tokens are its first T, and a count outside [0, a.T] means none
  const int T = a.T_dev ? live_tokens(a.T_dev, a.T) : a.T;
  const int H = a.H, E = a.E;
  if (a.T_dev && blockIdx.x == 0 && threadIdx.x == 0 && T != *a.T_dev)
    set_status(a.grp.status, STRATA_DEV_BAD_TOKENS);
  griddep_launch();  // the gate/up GEMM may launch now; it waits for this grid before reading
  const int wpe = kRsWarps / a.epc;  // warps per expert
  const int slot = warp / wpe, part = warp - slot * wpe;
  const int e = blockIdx.x * a.epc + slot;

  // logits: each warp dots its H slice of one router row with every token, 4 tokens x 4 vectors
  // of 8 columns per lane and pass, all loads of a pass in flight together
  const int nvec = H / 8;
  const int vb = part * nvec / wpe, ve = (part + 1) * nvec / wpe;
  const int64_t wro = static_cast<int64_t>(e < E ? e : 0) * H;
  const float4* wrow = reinterpret_cast<const float4*>(static_cast<const float*>(a.wr) + wro);
  const uint4* wrow16 = reinterpret_cast<const uint4*>(static_cast<const __half*>(a.wr) + wro);
  const uint4* xv = reinterpret_cast<const uint4*>(a.x);
  const uint64_t pol = l2_evict_first_policy();  // the router rows are read once per call
  constexpr int TB = 8;  // tokens per pass: every load of a pass is in flight together
  // the warps of expert slot 0 read all of x: they also find each token's largest magnitude,
  // from which the f16 copy of x gets its range exponent
  __shared__ uint32_t xmag[kRsWarps][kRouteSmallMaxT];
  __shared__ int xexp_s[kRouteSmallMaxT];
  for (int t0 = 0; t0 < T; t0 += TB) {
    float acc[TB] = {};
    uint32_t mag[TB] = {};
    if (e < E) {
      for (int v0 = vb + lane; v0 < ve; v0 += 128) {
        float4 w[4][2];
        uint4 xr[TB][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int v = v0 + 32 * i;
          if (v < ve) {
            if (kF16) {
              const uint4 hv = ldg_hint(wrow16 + v, pol);
              const __half2* h2 = reinterpret_cast<const __half2*>(&hv);
              const float2 f0 = __half22float2(h2[0]), f1 = __half22float2(h2[1]);
              const float2 f2 = __half22float2(h2[2]), f3 = __half22float2(h2[3]);
              w[i][0] = make_float4(f0.x, f0.y, f1.x, f1.y);
              w[i][1] = make_float4(f2.x, f2.y, f3.x, f3.y);
            } else {
              const uint4 u0 = ldg_hint(reinterpret_cast<const uint4*>(wrow + 2 * v), pol);
              const uint4 u1 = ldg_hint(reinterpret_cast<const uint4*>(wrow + 2 * v + 1), pol);
              w[i][0] = make_float4(__uint_as_float(u0.x), __uint_as_float(u0.y),
                                    __uint_as_float(u0.z), __uint_as_float(u0.w));
              w[i][1] = make_float4(__uint_as_float(u1.x), __uint_as_float(u1.y),
                                    __uint_as_float(u1.z), __uint_as_float(u1.w));
            }
#pragma unroll
            for (int tt = 0; tt < TB; ++tt)
              if (t0 + tt < T) xr[tt][i] = __ldg(xv + static_cast<int64_t>(t0 + tt) * nvec + v);
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (v0 + 32 * i >= ve) continue;
          const float wf[8] = {w[i][0].x, w[i][0].y, w[i][0].z, w[i][0].w,
                               w[i][1].x, w[i][1].y, w[i][1].z, w[i][1].w};
#pragma unroll
          for (int tt = 0; tt < TB; ++tt) {
            if (t0 + tt >= T) continue;
            if (slot == 0) mag[tt] = max(mag[tt], bf16x8_mag(xr[tt][i]));
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&xr[tt][i]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 f = __bfloat1622float2(p[q]);
              acc[tt] = fmaf(f.x, wf[2 * q], acc[tt]);
              acc[tt] = fmaf(f.y, wf[2 * q + 1], acc[tt]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < TB; ++tt) {
      float v = acc[tt];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && t0 + tt < T) red[warp][t0 + tt] = v;
      if (a.x_f16 && slot == 0) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, mag[tt]);
        if (lane == 0 && t0 + tt < T) xmag[part][t0 + tt] = m;
      }
    }
  }
  __syncthreads();
  // the H slices of one expert, summed in slice order
  for (int i = threadIdx.x; i < a.epc * T; i += blockDim.x) {
    const int sl = i / T, t = i - sl * T;
    const int ee = blockIdx.x * a.epc + sl;
    if (ee >= E) continue;
    float v = 0.f;
    for (int p = 0; p < wpe; ++p) v += red[sl * wpe + p][t];
    if (a.bias) v += a.bias[ee];
    a.logits[static_cast<int64_t>(t) * E + ee] = v;
  }
  // The decode grouped GEMM reads x with every 8-wide chunk pair-interleaved (as f16 for the
  // CTA-staged kernel, bf16 for the per-warp one). Only the GEMMs, which wait for this grid, read
  // the copy, so the CTAs that do not take part in the top-k make it after signalling their logits
  // (off the top-k's path); with no such CTA every CTA copies first.
  auto copy_x = [&](int part, int nparts) {
    if (a.x_f16) {
      // each token's range exponent, from the magnitudes found by the expert-slot-0 warps; the
      // copying CTA of part 0 publishes them for the GEMMs
      for (int t = threadIdx.x; t < T; t += blockDim.x) {
        uint32_t m = 0;
        for (int p = 0; p < wpe; ++p) m = max(m, xmag[p][t]);
        xexp_s[t] = range_exp(m);
        if (part == 0 && a.xexp) a.xexp[t] = xexp_s[t];
      }
      __syncthreads();
    }
    const int nv = T * (H / 8);
    for (int i = part * blockDim.x + threadIdx.x; i < nv; i += nparts * blockDim.x) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
      uint4 o;
      if (a.x_f16) {
        o = bf16_chunk_to_f16_pairs(v, exp2i(-xexp_s[i / (H / 8)]));
      } else {
        o.x = prmt(v.x, v.z, 0x5410);
        o.y = prmt(v.x, v.z, 0x7632);
        o.z = prmt(v.y, v.w, 0x5410);
        o.w = prmt(v.y, v.w, 0x7632);
      }
      reinterpret_cast<uint4*>(a.x_perm)[i] = o;
    }
  };

  // The last G CTAs to finish their logits (G = one warp per token, 8 tokens per CTA) wait for
  // the others, take the top-k of their tokens, and the last of them groups the rows. With one
  // such CTA (T <= 8) the ids stay in its shared memory.
  __shared__ int role_s, arrival_s;
  // (at least one: with no live token it still writes the empty grouping the GEMMs read)
  const int G = min(static_cast<int>(gridDim.x), max(1, (T + kRsWarps - 1) / kRsWarps));
  const int ncopy = static_cast<int>(gridDim.x) - G;  // CTAs outside the top-k
  if (a.x_perm && ncopy == 0) copy_x(blockIdx.x, gridDim.x);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&a.grp.hdr->route_done, 1u);
    arrival_s = static_cast<int>(prev);
    int r = static_cast<int>(prev) - ncopy;
    // wait (bounded, ~1 s) for the CTAs still writing logits: all of them run already (this
    // grid's dependents launch only once every CTA of it has started); on time-out this CTA
    // gives up its top-k and the status tells the host
    if (r >= 0 && prev != gridDim.x - 1 &&
        !spin_until_geq(&a.grp.hdr->route_done, gridDim.x, kRouterWaitCycles, a.grp.status))
      r = -1;
    role_s = r;
  }
  __syncthreads();
  const int role = role_s;
  if (role < 0) {
    // arrivals 0 .. ncopy-1 are exactly the CTAs outside the top-k: each copies its share of x
    if (a.x_perm && arrival_s < ncopy) copy_x(arrival_s, ncopy);
    return;
  }
  __threadfence();

  int* s_ids = reinterpret_cast<int*>(rs_smem + route_small_ids_off(a));
  float* s_gates = reinterpret_cast<float*>(s_ids + T * a.k);
  if (G == 1) {
    // tokens warp, warp + 8, ... (up to 4 at once per warp), logits read from L2 into registers
    const int tpw = T <= kRsWarps ? 1 : (T <= 2 * kRsWarps || E > 512) ? 2 : 4;
#pragma unroll 1
    for (int t0 = warp; t0 < T; t0 += kRsWarps * tpw) {
      if (tpw == 1)
        warp_softmax_topk<1, true>(a.logits, E, t0, kRsWarps, T, E, a.k, a.flags, s_ids, s_gates);
      else if (tpw == 2)
        warp_softmax_topk<2, true>(a.logits, E, t0, kRsWarps, T, E, a.k, a.flags, s_ids, s_gates);
      else
        warp_softmax_topk<4, true>(a.logits, E, t0, kRsWarps, T, E, a.k, a.flags, s_ids, s_gates);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < T * a.k; i += blockDim.x) {
      a.ids[i] = s_ids[i];
      a.gates[i] = s_gates[i];
    }
  } else {
    // one token per warp: token role * 8 + warp, results straight to global memory
    const int t = role * kRsWarps + warp;
    if (t < T) warp_softmax_topk<1, true>(a.logits, E, t, 1, T, E, a.k, a.flags, a.ids, a.gates);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned prev = atomicAdd(&a.grp.hdr->topk_done, 1u);
      role_s = (prev == static_cast<unsigned>(G) - 1u) ? 1 : 0;
    }
    __syncthreads();
    if (!role_s) return;
    __threadfence();
    for (int i = threadIdx.x; i < T * a.k; i += blockDim.x) s_ids[i] = __ldcg(a.ids + i);
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    a.grp.hdr->route_done = 0;
    a.grp.hdr->topk_done = 0;
  }
  if (a.do_group) {
    PermuteArgs g = a.grp;
    g.T = T;
    if (route_small_compact_group(a))
      group_rows_small<kRsWarps>(g, s_ids, reinterpret_cast<int*>(rs_smem));
    else
      group_rows<kRsWarps>(g, s_ids, carve_group_smem(reinterpret_cast<int*>(rs_smem), kRsWarps, E));
  }
}

cudaError_t launch_route_small(const RouteSmallArgs& a, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const dim3 grid((a.E + a.epc - 1) / a.epc);
  const size_t smem = route_small_smem(a);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(route_small_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(route_small_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  if (a.wr_fp16)
    route_small_kernel<true><<<grid, kRsWarps * 32, smem, stream>>>(a);
  else
    route_small_kernel<false><<<grid, kRsWarps * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- large batches

// Large batches on tensor cores: logits = x Wr^T with Wr split exactly into three bf16 parts
// (hi + mid + lo == the fp32 value; two parts for an fp16 router: 8 + 3 significant bits), so
// every product x*part is exact and the mma.sync fp32 accumulation matches an fp32 GEMM. Tile 64 tokens x 64 experts, 8 warps (2 x 4), warp tile
// 32 x 16; contraction staged 32 columns at a time (double-buffered cp.async for x, registers for
// the fp32 router tile, split on the way into shared memory); every 256 columns the chunk sum joins
// the running total with compensated (Kahan) addition. Split along H (blockIdx.z) like the SIMT
// kernel so that small grids still fill the GPU.
constexpr int kRtT = 64, kRtE = 64, kRtK = 32, kRtPad = 40;  // shared rows padded to 80 bytes

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1]) : "r"(a));
}

template <bool kF16>
__global__ void __launch_bounds__(256) router_logits_tc_kernel(const __nv_bfloat16* __restrict__ x,
                                                               const void* __restrict__ wr_, int T,
                                                               int H, int E, int h_per_split,
                                                               float* __restrict__ partial) {
  constexpr int NSPLIT = kF16 ? 2 : 3;
  __shared__ __align__(16) __nv_bfloat16 xs[2][kRtT][kRtPad];
  __shared__ __align__(16) __nv_bfloat16 ws[3][kRtE][kRtPad];  // hi, mid, lo
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e0 = blockIdx.x * kRtE, t0 = blockIdx.y * kRtT;
  const int hbeg = blockIdx.z * h_per_split;
  const int hend = min(H, hbeg + h_per_split);
  const int wt = (warp >> 2) * 32;  // warp's token offset in the tile
  const int we = (warp & 3) * 16;   // warp's expert offset
  float acc[2][2][4] = {}, comp[2][2][4] = {}, part[2][2][4] = {};

  // x tile: 64 rows x 32 bf16 = 256 x 16 bytes, one cp.async per thread
  const int xr = tid >> 2, xc = (tid & 3) * 8;
  const bool xok = t0 + xr < T;
  const __nv_bfloat16* xsrc = x + static_cast<int64_t>(xok ? t0 + xr : 0) * H + xc;
  // router tile: 64 experts x 32 fp32 = 8 floats per thread
  const int wrr = tid >> 2, wc = (tid & 3) * 8;
  const bool wok = e0 + wrr < E;
  const int64_t woff = static_cast<int64_t>(wok ? e0 + wrr : 0) * H + wc;

  auto stage_x = [&](int buf, int hc) { cp_async16(&xs[buf][xr][xc], xsrc + hc, xok); };
  auto stage_w = [&](int hc) {
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (wok) {
      if (kF16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __half*>(wr_) + woff + hc));
        const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 ff = __half22float2(h2[i]);
          f[2 * i] = ff.x;
          f[2 * i + 1] = ff.y;
        }
      } else {
        const float* wsrc = static_cast<const float*>(wr_) + woff + hc;
        const float4 a = __ldg(reinterpret_cast<const float4*>(wsrc));
        const float4 b = __ldg(reinterpret_cast<const float4*>(wsrc) + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
      }
    }
    __nv_bfloat16 hi[8], mid[8], lo[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // f = hi + mid + lo exactly (24 = 8 + 8 + 8 significant bits)
      hi[i] = __float2bfloat16_rn(f[i]);
      const float r1 = f[i] - __bfloat162float(hi[i]);
      mid[i] = __float2bfloat16_rn(r1);
      lo[i] = __float2bfloat16_rn(r1 - __bfloat162float(mid[i]));
    }
    *reinterpret_cast<uint4*>(&ws[0][wrr][wc]) = *reinterpret_cast<uint4*>(hi);
    *reinterpret_cast<uint4*>(&ws[1][wrr][wc]) = *reinterpret_cast<uint4*>(mid);
    if (!kF16) *reinterpret_cast<uint4*>(&ws[2][wrr][wc]) = *reinterpret_cast<uint4*>(lo);
  };

  int buf = 0;
  if (hbeg < hend) stage_x(0, hbeg);
  cp_async_commit();
  int chunk_cols = 0;
  for (int hc = hbeg; hc < hend; hc += kRtK) {
    if (hc + kRtK < hend) stage_x(buf ^ 1, hc + kRtK);
    cp_async_commit();
    stage_w(hc);
    cp_async_wait<1>();
    __syncthreads();
#pragma unroll
    for (int ks = 0; ks < kRtK; ks += 16) {
      uint32_t a[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
        ldmatrix_x4(a[mi], &xs[buf][wt + mi * 16 + (lane & 15)][ks + (lane >> 4) * 8]);
#pragma unroll
      for (int sp = 0; sp < NSPLIT; ++sp) {
#pragma unroll
        for (int ni = 0; ni < 2; ++ni) {
          uint32_t b[2];
          ldmatrix_x2(b, &ws[sp][we + ni * 8 + (lane & 7)][ks + ((lane >> 3) & 1) * 8]);
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) mma_bf16_16816(part[mi][ni], a[mi], b[0], b[1], part[mi][ni]);
        }
      }
    }
    chunk_cols += kRtK;
    if (chunk_cols == 256 || hc + kRtK >= hend) {  // join the running total (compensated)
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 2; ++ni)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float y = part[mi][ni][c] - comp[mi][ni][c];
            const float t = acc[mi][ni][c] + y;
            comp[mi][ni][c] = (t - acc[mi][ni][c]) - y;
            acc[mi][ni][c] = t;
            part[mi][ni][c] = 0.f;
          }
      chunk_cols = 0;
    }
    __syncthreads();
    buf ^= 1;
  }
  cp_async_wait<0>();
  // C fragment: rows (tokens) lane/4 and lane/4 + 8, columns (experts) 2*(lane%4) + {0,1}
  float* out = partial + static_cast<int64_t>(blockIdx.z) * T * E;
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 2; ++ni)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int t = t0 + wt + mi * 16 + (lane >> 2) + (c >= 2 ? 8 : 0);
        const int e = e0 + we + ni * 8 + 2 * (lane & 3) + (c & 1);
        if (t < T && e < E) out[static_cast<int64_t>(t) * E + e] = acc[mi][ni][c];
      }
}

// One warp per token; the split partials are summed in split order.
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ partial,
                                                          int nsplit, const float* __restrict__ bias,
                                                          int T, int E, int k, uint32_t flags,
                                                          int* __restrict__ ids,
                                                          float* __restrict__ gates) {
  extern __shared__ float lg_all[];  // [8 warps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float* lg = lg_all + warp * E;
  for (int e = lane; e < E; e += 32) {
    float v = 0.f;
    for (int s = 0; s < nsplit; ++s) v += __ldcg(partial + (static_cast<int64_t>(s) * T + t) * E + e);
    if (bias) v += bias[e];
    lg[e] = v;
  }
  __syncwarp();
  warp_softmax_topk<1, false>(lg, E, 0, 1, 1, E, k, flags, ids + static_cast<int64_t>(t) * k,
                              gates + static_cast<int64_t>(t) * k);
}

int router_num_splits(int64_t T, int64_t H, int E, int num_sms) {
  const int64_t tiles = ((E + kRtE - 1) / kRtE) * ((T + kRtT - 1) / kRtT);
  int64_t want = (num_sms + tiles - 1) / tiles;  // about one CTA per SM
  const int64_t max_split = H / 128;
  if (want > max_split) want = max_split;
  if (want > 16) want = 16;
  if (want < 1) want = 1;
  return static_cast<int>(want);
}

cudaError_t launch_router(const void* x, const void* wr, const float* bias, int64_t T, int64_t H,
                          int E, int k, uint32_t flags, int nsplit, float* partial, int* ids,
                          float* gates, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  // splits cover whole 128-column groups (a multiple of the 32-wide chunk)
  const int64_t groups = H / 128;
  const int64_t gps = (groups + nsplit - 1) / nsplit;
  const int h_per_split = static_cast<int>(gps * 128);
  const int used = static_cast<int>((groups + gps - 1) / gps);
  dim3 grid((E + kRtE - 1) / kRtE, static_cast<unsigned>((T + kRtT - 1) / kRtT), used);
  if (flags & STRATA_ROUTER_FP16)
    router_logits_tc_kernel<true><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                            wr, static_cast<int>(T),
                                                            static_cast<int>(H), E, h_per_split,
                                                            partial);
  else
    router_logits_tc_kernel<false><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                             wr, static_cast<int>(T),
                                                             static_cast<int>(H), E, h_per_split,
                                                             partial);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t smem = static_cast<size_t>(8) * E * sizeof(float);
  router_topk_kernel<<<static_cast<unsigned>((T + 7) / 8), 256, smem, stream>>>(
      partial, used, bias, static_cast<int>(T), E, k, flags, ids, gates);
  return cudaGetLastError();
}

}  // namespace strata
