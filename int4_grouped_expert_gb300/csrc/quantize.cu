// K1: symmetric group quantization ("Strata" MoE tuning notes, lpnh.cn/news/2730718, §2.1
// group_quantize sketch: scale = absmax / (2^(bits-1) - 1), codes = round(w / scale) clamped to
// the code range, 128 weights per group by default; 64 and 256 are accepted too). bits = 4 (the
// experts' width: range [-8, 7], two codes per byte, even k in the low nibble) or 8 (range
// [-128, 127], one code per byte).
//
// HBM-streaming pass: G/8 threads own one G-wide group (8 fp16 = one 16-byte load each), find the
// group's absmax with butterfly shuffles, and write 4 bytes of packed codes (8 for 8-bit codes)
// each (the group's codes are contiguous) plus one fp16 scale. Each thread walks its groups with
// a grid-stride loop, four groups' loads in flight at a time.
//
// Exactness: absmax / 7.0f (or / 127.0f) is an IEEE fp32 division rounded once more to fp16 (no
// double-rounding hazard: the exact quotient of an 11-bit significand by 7 or 127 is either exact
// in fp16 or at least 2^-18 relative away from every fp16 midpoint). The codes round w * (1/s)
// and settle exact ties with the exact residual w - q*s (see quantize_one), which gives
// round-half-even of the exact quotient w / s for every pair of fp16 values.
#include "kernels.cuh"

namespace strata {

// One group: TPG lanes hold 8 fp16 each. Codes: 4 bytes per lane (4-bit) or 8 (8-bit).
template <int TPG, int kBits>
__device__ __forceinline__ void quantize_one(const uint4& v, unsigned half_mask, int sub, int64_t g,
                                             void* __restrict__ codes,
                                             __half* __restrict__ scales, uint32_t* status) {
  constexpr float kQmax = kBits == 4 ? 7.0f : 127.0f;
  // |w| as fp16 bit patterns: their integer order is the order of the magnitudes, and any pattern
  // at or above 0x7C00 is inf or nan, so one integer max gives both absmax and finiteness
  const uint32_t m01 = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
  const uint32_t m23 = __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
  const uint32_t m2 = __vmaxu2(m01, m23);
  uint32_t mbits = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
  for (int o = TPG / 2; o > 0; o >>= 1) mbits = max(mbits, __shfl_xor_sync(half_mask, mbits, o));
  const bool finite = mbits < 0x7C00u;
  const float amax = finite ? __half2float(__ushort_as_half(static_cast<unsigned short>(mbits))) : 0.f;
  const __half* h = reinterpret_cast<const __half*>(&v);
  __half s_h = __float2half_rn(amax / kQmax);
  const float s = __half2float(s_h);
  uint32_t packed = 0, lo = 0, hi = 0;  // 4-bit: 8 nibbles; 8-bit: 8 bytes in (lo, hi)
  if (finite && s > 0.0f) {
    // q = RNE(w / s) without a division per weight: w * (1/s) rounds to the right integer except
    // at exact ties (for fp16 w and s, w/s is either a half-integer or at least 2^-13 away from
    // every half-integer, far more than the error of the fp32 product), and the residual
    // w - q*s, exact in fp32 (q*s has at most 8 + 11 significant bits), finds the ties: there it
    // is +-s/2 and q moves to the even neighbour.
    const float inv = 1.0f / s;
    const float half_s = 0.5f * s;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float wf = __half2float(h[i]);
      float q = rintf(wf * inv);
      const float r = fmaf(-q, s, wf);
      if (static_cast<int>(q) & 1) q += r == half_s ? 1.0f : (r == -half_s ? -1.0f : 0.0f);
      q = fminf(fmaxf(q, -kQmax - 1.0f), kQmax);
      const uint32_t c = static_cast<uint32_t>(static_cast<int>(q));
      if (kBits == 4)
        packed |= (c & 0xFu) << (4 * i);
      else if (i < 4)
        lo |= (c & 0xFFu) << (8 * i);
      else
        hi |= (c & 0xFFu) << (8 * (i - 4));
    }
  }
  if (!finite) {
    s_h = __ushort_as_half(0x7E00);  // NaN scale marks the group
    if (sub == 0) set_status(status, STRATA_DEV_NONFINITE);
  }
  if (kBits == 4)
    __stcs(static_cast<uint32_t*>(codes) + g * TPG + sub, packed);
  else
    __stcs(static_cast<uint2*>(codes) + g * TPG + sub, make_uint2(lo, hi));
  if (sub == 0) scales[g] = s_h;
}

// Each TPG-lane team walks groups g, g + stride, ... with four groups' loads in flight at a time.
template <int TPG, int kBits>
__global__ void __launch_bounds__(256) quantize_groups_kernel(const uint4* __restrict__ w,
                                                              int64_t n_groups,
                                                              void* __restrict__ codes,
                                                              __half* __restrict__ scales,
                                                              uint32_t* status) {
  const int sub = threadIdx.x & (TPG - 1);  // position in the group
  // the teams of a warp may leave the loop at different times: shuffle within the team only
  const unsigned team_mask =
      TPG == 32 ? 0xFFFFFFFFu : (((1u << TPG) - 1u) << (threadIdx.x & 31 & ~(TPG - 1)));
  const int64_t first = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / TPG;
  const int64_t stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) / TPG;
  constexpr int U = 4;
  for (int64_t g0 = first; g0 < n_groups; g0 += U * stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = g0 + u * stride;
      if (g < n_groups) v[u] = __ldcs(w + g * TPG + sub);  // streaming: every weight read once
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = g0 + u * stride;
      if (g < n_groups) quantize_one<TPG, kBits>(v[u], team_mask, sub, g, codes, scales, status);
    }
  }
}

cudaError_t launch_quantize(const void* w, int64_t n, int64_t k, int group, int bits,
                            uint8_t* codes, void* scales, uint32_t* status, cudaStream_t stream,
                            int num_sms) {
  const int64_t n_groups = n * (k / group);
  if (n_groups == 0) return cudaSuccess;
  const int threads = 256;
  const int tpg = group / 8;                     // threads per group
  int64_t blocks = (n_groups * tpg + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // ~8 resident blocks/SM, grid-stride
  if (blocks > cap) blocks = cap;
  const uint4* wv = static_cast<const uint4*>(w);
  __half* sv = static_cast<__half*>(scales);
  const unsigned b = static_cast<unsigned>(blocks);
#define STRATA_Q(T, B) quantize_groups_kernel<T, B><<<b, threads, 0, stream>>>(wv, n_groups, codes, sv, status)
  if (bits == 4) {
    if (tpg == 8) STRATA_Q(8, 4);
    else if (tpg == 16) STRATA_Q(16, 4);
    else if (tpg == 32) STRATA_Q(32, 4);
    else return cudaErrorInvalidValue;
  } else if (bits == 8) {
    if (tpg == 8) STRATA_Q(8, 8);
    else if (tpg == 16) STRATA_Q(16, 8);
    else if (tpg == 32) STRATA_Q(32, 8);
    else return cudaErrorInvalidValue;
  } else {
    return cudaErrorInvalidValue;
  }
#undef STRATA_Q
  return cudaGetLastError();
}

}  // namespace strata
