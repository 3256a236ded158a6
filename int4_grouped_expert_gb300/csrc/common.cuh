// Shared device helpers of the strata kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/strata.h"

namespace strata {

constexpr int kGroup = STRATA_GROUP;  // weights per scale group

// Workspace header (first 256 bytes of every route/forward workspace).
struct WsHeader {
  uint32_t status;      // STRATA_DEV_* bits
  int32_t nseg;         // active expert segments (the shared one first, then routed experts with rows)
  int32_t n_items_gu;   // gate/up work items
  int32_t n_items_dn;   // down work items
  int32_t next_gu;      // dynamic scheduler: next gate/up item
  int32_t next_dn;      // dynamic scheduler: next down item
  uint32_t route_done;  // CTAs of the fused router that finished their logits
  int32_t n_chunks;     // warp path: 8-row chunks in the chunk list
  uint32_t topk_done;   // CTAs of the fused router that finished their share of the top-k
  int32_t pad[55];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

__device__ __forceinline__ void set_status(uint32_t* st, uint32_t bits) {
  if (st) atomicOr(st, bits);
}

// Spin until the device-scope counter reaches `target`, giving up after `limit` SM clocks: then
// the status gets STRATA_DEV_TIMEOUT and the result is false.
__device__ __forceinline__ bool spin_until_geq(const unsigned* ctr, unsigned target,
                                               long long limit, uint32_t* status) {
  const long long t0 = clock64();
  while (*reinterpret_cast<const volatile unsigned*>(ctr) < target) {
    __nanosleep(64);
    if (clock64() - t0 > limit) {
      set_status(status, STRATA_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Live tokens of a fixed-size batch whose count sits in device memory: the count itself when it
// lies in [0, max], else 0 (the caller flags STRATA_DEV_BAD_TOKENS).
__device__ __forceinline__ int live_tokens(const int* count, int max) {
  const int t = *reinterpret_cast<const volatile int*>(count);
  return (t >= 0 && t <= max) ? t : 0;
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

// ---------------------------------------------------------------------------- mma.sync bf16
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C (fp32).
// D = A * B + C, m16n8k16, f16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// ---------------------------------------------------------------------------- int4 -> bf16
// A 32-bit word holds 8 codes, nibble i = element i (4-bit two's complement). After flipping the
// sign bit of every nibble (w ^ 0x88888888 turns q into q + 8 in [0, 15]), OR-ing a nibble into the
// low mantissa bits of bf16 128.0 (0x4300) gives exactly 128 + q + 8; subtracting 136 leaves q.
// pair(w, i) returns bf16x2 {element i, element i + 4} (low half first).
__device__ __forceinline__ uint32_t int4pair_to_bf16x2(uint32_t w_offset_binary, int i) {
  uint32_t v = (w_offset_binary >> (4 * i)) & 0x000F000Fu;
  v |= 0x43004300u;
  __nv_bfloat162 r = *reinterpret_cast<__nv_bfloat162*>(&v);
  const __nv_bfloat162 bias = __floats2bfloat162_rn(136.0f, 136.0f);
  r = __hsub2(r, bias);  // exact: small integers
  return *reinterpret_cast<uint32_t*>(&r);
}

// Byte permute: result bytes selected from {a (bytes 0-3), b (bytes 4-7)}.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// ---------------------------------------------------------------------------- cp.async
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  int sz = pred ? 16 : 0;  // zero-fill when the source row does not exist
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// L2 policy for data a kernel streams once per call (expert weights and scales, router weights):
// evicted before normal lines, so that the layer's small reused state (code, activations,
// routing buffers) stays in L2 while hundreds of MB of weights pass through it.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// 16-byte read-only load with an L2 policy.
__device__ __forceinline__ uint4 ldg_hint(const uint4* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// Two fp32 values as an f16x2 word (lo in the low half), rounded to nearest and saturated to
// +-65504 (finite inputs never become inf; NaN stays NaN).
__device__ __forceinline__ uint32_t f32x2_to_f16x2_sat(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ __half f32_to_f16_sat(float x) {
  unsigned short d;
  asm("cvt.rn.satfinite.f16.f32 %0, %1;" : "=h"(d) : "f"(x));
  return __ushort_as_half(d);
}
// The two bf16 values of a word as fp32 (exact), low half first.
__device__ __forceinline__ float bf16_lo_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
// One 8-wide chunk of bf16 activations (natural order, words (x0,x1) (x2,x3) (x4,x5) (x6,x7)) as
// f16 in the order the CTA-staged decode GEMM reads: words (x0,x4) (x2,x6) (x1,x5) (x3,x7), i.e.
// element i of the chunk at position bitrev3(i). A 16-byte load then gives the two B-operand
// register pairs of one MMA step in adjacent registers.
// s: an exact power of two that the values are multiplied by first (see range_exp).
__device__ __forceinline__ uint4 bf16_chunk_to_f16_pairs(uint4 v, float s = 1.0f) {
  uint4 o;
  o.x = f32x2_to_f16x2_sat(bf16_lo_f32(v.x) * s, bf16_lo_f32(v.z) * s);
  o.y = f32x2_to_f16x2_sat(bf16_lo_f32(v.y) * s, bf16_lo_f32(v.w) * s);
  o.z = f32x2_to_f16x2_sat(bf16_hi_f32(v.x) * s, bf16_hi_f32(v.z) * s);
  o.w = f32x2_to_f16x2_sat(bf16_hi_f32(v.y) * s, bf16_hi_f32(v.w) * s);
  return o;
}

// Range of the f16 GEMM operands. A row of activations (x, or h) whose magnitude would leave the
// f16 range is stored as act * 2^-e (an exact power of two: no rounding is added except to
// values that become f16 subnormals, far below the row's largest entries), and the GEMM that reads
// it multiplies its fp32 result by 2^e. e = 0 for every row whose entries stay below 16, so
// ordinary inputs are untouched; rows of a residual stream that has grown without normalisation
// are the ones that need it.
//
// 2^n as a float, exactly, for -126 <= n <= 127.
__device__ __forceinline__ float exp2i(int n) { return __int_as_float((n + 127) << 23); }
// Largest magnitude among 8 bf16 values as an integer key (bf16 bits without the sign: their
// integer order is the order of the magnitudes).
__device__ __forceinline__ uint32_t bf16x8_mag(uint4 v) {
  const uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                              __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}
// The row exponent for a largest bf16 magnitude (key as above): the smallest e >= 0 with
// max * 2^-e < 16, capped at 60 (so that 2e stays a float exponent).
__device__ __forceinline__ int range_exp(uint32_t mag_key) {
  const int e = static_cast<int>(mag_key >> 7) - 127;  // max in [2^e, 2^(e+1))
  return e < 4 ? 0 : min(e - 3, 60);
}

// silu(u) = u * sigmoid(u) with the fast exp and divide intrinsics (a few ulp of fp32: the result
// is rounded to bf16 right after). Large negative u: exp overflows to inf and the quotient is 0.
__device__ __forceinline__ float silu_f(float u) { return __fdividef(u, 1.0f + __expf(-u)); }
// silu(u_s * up) / up for a power of two up: the SiLU of a value held as u_s = u / up, returned
// at the same scale (u_s * sigmoid(u)); equal to silu_f(u_s) when up = 1.
__device__ __forceinline__ float silu_scaled(float u_s, float up) {
  return __fdividef(u_s, 1.0f + __expf(-u_s * up));
}

// Programmatic dependent launch: a kernel launched with the PDL attribute may start while its
// predecessor in the stream still runs; griddep_wait() blocks until the predecessor grid has
// completed and its memory is visible (a no-op without the attribute). griddep_launch() lets the
// next kernel start launching early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace strata
