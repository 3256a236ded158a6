// K1: symmetric group quantization ("Strata" MoE tuning notes, lpnh.cn/news/2730718, §2.1
// group_quantize sketch: scale = absmax / (2^(bits-1) - 1), codes = round(w / scale) clamped to
// the code range, 128 weights per group by default; 64 and 256 are accepted too). bits = 4 (the
// experts' width: range [-8, 7], two codes per byte, even k in the low nibble) or 8 (range
// [-128, 127], one code per byte).
//
// HBM-streaming pass: G/16 threads own one G-wide group (16 fp16 = two 16-byte loads each), find
// the group's absmax with butterfly shuffles, and write 8 bytes of packed codes (16 for 8-bit
// codes) each (the group's codes are contiguous) plus one fp16 scale. Each thread walks its groups
// with a grid-stride loop, two groups' loads in flight at a time. The pass is bound by issue, not
// by DRAM, so the per-weight work is a handful of fp32 instructions (see quantize_one).
//
// Exactness: the scale is absmax times the fp32 reciprocal of 7 (127) rounded to fp16, which is
// the fp16 rounding of the exact quotient for every fp16 absmax (checked exhaustively: the
// quotient is never closer than 2^-14.8 relative to an fp16 midpoint, 2^-18.9 for 127). The codes
// round w * (1/s) with one fma and settle exact ties with the exact residual w - q*s (see
// quantize_one), which gives round-half-even of the exact quotient w / s for every pair of fp16
// values.
#include "kernels.cuh"

namespace strata {

// One group: TPG lanes hold 16 fp16 each (two 16-byte loads). Codes: 8 bytes per lane (4-bit)
// or 16 (8-bit).
template <int TPG, int kBits>
__device__ __forceinline__ void quantize_one(const uint4 (&v)[2], unsigned team_mask, int sub,
                                             int64_t g, void* __restrict__ codes,
                                             __half* __restrict__ scales, uint32_t* status) {
  constexpr float kQmax = kBits == 4 ? 7.0f : 127.0f;
  constexpr float kInvQmax = 1.0f / kQmax;     // fp32 1/7 (1/127), rounded once
  constexpr float kMagic = 12582912.0f;        // 1.5 * 2^23: adding it rounds to an integer
  constexpr uint32_t kCodeMask = kBits == 4 ? 0xFu : 0xFFu;
  // |w| as fp16 bit patterns: their integer order is the order of the magnitudes, and any pattern
  // at or above 0x7C00 is inf or nan, so one integer max gives both absmax and finiteness
  uint32_t m2 = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    m2 = __vmaxu2(m2, __vmaxu2(v[j].x & 0x7FFF7FFFu, v[j].y & 0x7FFF7FFFu));
    m2 = __vmaxu2(m2, __vmaxu2(v[j].z & 0x7FFF7FFFu, v[j].w & 0x7FFF7FFFu));
  }
  uint32_t mbits = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
  for (int o = TPG / 2; o > 0; o >>= 1) mbits = max(mbits, __shfl_xor_sync(team_mask, mbits, o));
  const bool finite = mbits < 0x7C00u;
  const float amax = finite ? __half2float(__ushort_as_half(static_cast<unsigned short>(mbits))) : 0.f;
  // scale = fp16(absmax / qmax): the product with the rounded reciprocal rounds to the same fp16
  // as the exact quotient for every fp16 absmax (that quotient is at least 2^-14.8 relative away
  // from every fp16 rounding midpoint, the product within 2^-23 of it)
  __half s_h = __float2half_rn(amax * kInvQmax);
  const float s = __half2float(s_h);
  const __half2* h2 = reinterpret_cast<const __half2*>(&v[0]);
  const __half* h1 = reinterpret_cast<const __half*>(&v[0]);
  // packed codes: weight i at bits 4i of word i/8 (4-bit), 8i of word i/4 (8-bit)
  constexpr int kWords = kBits == 4 ? 2 : 4;
  uint32_t out[kWords];
#pragma unroll
  for (int j = 0; j < kWords; ++j) out[j] = 0u;
  // bits of q + kMagic hold q in two's complement in their low bits
  auto put = [&](int i, uint32_t qbits) {
    if (kBits == 4) out[i >> 3] |= (qbits & kCodeMask) << (4 * (i & 7));
    else out[i >> 2] |= (qbits & kCodeMask) << (8 * (i & 3));
  };
  if (finite && s >= 6.103515625e-05f) {
    // A normal fp16 scale is within 2^-11 relative of absmax / qmax, so |w / s| <=
    // qmax / (1 - 2^-11) < qmax + 1/2 and q needs no clamp. q = RNE(w / s) without a division
    // per weight: fma(w, 1/s, kMagic) rounds w/s to the right integer except at exact ties (for
    // fp16 w and s, w/s is either a half-integer or at least 2^-13 away from every half-integer,
    // far more than the error of w * (1/s) with a reciprocal good to a few ulp); the residual
    // w - q*s, exact in fp32 (q*s has at most 8 + 11 significant bits), finds the ties: there it
    // is +-s/2, and q moves to the even neighbour.
    float inv;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(s));
    const float half_s = 0.5f * s;
    bool tie = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 wf = __half22float2(h2[i]);
      const float f0 = fmaf(wf.x, inv, kMagic), f1 = fmaf(wf.y, inv, kMagic);
      const float r0 = fmaf(kMagic - f0, s, wf.x), r1 = fmaf(kMagic - f1, s, wf.y);
      tie |= (fabsf(r0) == half_s) | (fabsf(r1) == half_s);
      put(2 * i, __float_as_uint(f0));
      put(2 * i + 1, __float_as_uint(f1));
    }
    if (tie) {  // rare: redo the lane's weights, settling exact ties to the even code
#pragma unroll
      for (int j = 0; j < kWords; ++j) out[j] = 0u;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float wf = __half2float(h1[i]);
        float q = fmaf(wf, inv, kMagic) - kMagic;
        const float r = fmaf(-q, s, wf);
        if ((static_cast<int>(q) & 1) && fabsf(r) == half_s) q += r > 0.f ? 1.0f : -1.0f;
        put(i, __float_as_uint(q + kMagic));
      }
    }
  } else if (finite && s > 0.0f) {
    // subnormal scale: the exact quotient, clamped (a subnormal scale can push |w / s| past qmax)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float q = rintf(__half2float(h1[i]) / s);
      q = fminf(fmaxf(q, -kQmax - 1.0f), kQmax);
      put(i, __float_as_uint(q + kMagic));
    }
  }  // else: scale 0 or a non-finite group, codes 0
  if (!finite) {
    s_h = __ushort_as_half(0x7E00);  // NaN scale marks the group
    if (sub == 0) set_status(status, STRATA_DEV_NONFINITE);
  }
  if (kBits == 4)
    __stcs(static_cast<uint2*>(codes) + g * TPG + sub, make_uint2(out[0], out[1]));
  else
    __stcs(static_cast<uint4*>(codes) + g * TPG + sub, make_uint4(out[0], out[1], out[2], out[3]));
  if (sub == 0) scales[g] = s_h;
}

// Each TPG-lane team walks groups g, g + stride, ... with two groups' loads in flight at a time.
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
  constexpr int U = 2;
  for (int64_t g0 = first; g0 < n_groups; g0 += U * stride) {
    uint4 v[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = g0 + u * stride;
      if (g < n_groups) {  // streaming: every weight is read once
        const uint4* src = w + (g * TPG + sub) * 2;
        v[u][0] = __ldcs(src);
        v[u][1] = __ldcs(src + 1);
      }
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
  const int tpg = group / 16;                    // threads per group (16 weights each)
  int64_t blocks = (n_groups * tpg + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;  // ~8 resident blocks/SM, grid-stride
  if (blocks > cap) blocks = cap;
  const uint4* wv = static_cast<const uint4*>(w);
  __half* sv = static_cast<__half*>(scales);
  const unsigned b = static_cast<unsigned>(blocks);
#define STRATA_Q(T, B) quantize_groups_kernel<T, B><<<b, threads, 0, stream>>>(wv, n_groups, codes, sv, status)
  if (bits == 4) {
    if (tpg == 4) STRATA_Q(4, 4);
    else if (tpg == 8) STRATA_Q(8, 4);
    else if (tpg == 16) STRATA_Q(16, 4);
    else return cudaErrorInvalidValue;
  } else if (bits == 8) {
    if (tpg == 4) STRATA_Q(4, 8);
    else if (tpg == 8) STRATA_Q(8, 8);
    else if (tpg == 16) STRATA_Q(16, 8);
    else return cudaErrorInvalidValue;
  } else {
    return cudaErrorInvalidValue;
  }
#undef STRATA_Q
  return cudaGetLastError();
}

}  // namespace strata
