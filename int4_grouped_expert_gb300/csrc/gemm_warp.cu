// K4 (warp path): W4A16 grouped GEMM for segments with few rows — decode, where the layer is bound
// by streaming the activated experts' int4 weights from HBM. One launch covers every expert's
// group ("Strata" 3090 tuning, xdnf.cn/news/329730, §3.2: one grouped GEMM instead of one GEMM
// launch per expert); dequantization happens in registers ("Strata" architecture essay,
// dpshk.com/news/6309482, §3.2: decode is bandwidth-bound, so use wide vector loads and keep the
// small operands close).
//
// Work item = (segment, 16 weight rows, up to 8 token rows). A warp computes it with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) and swapped operands: the 16 weight rows are the
// A operand, the token rows the 8-wide B operand.
//  * The int4 codes are read in their canonical row-major layout. Lane (g = lane/4, t = lane%4)
//    loads 16 bytes = 32 codes of rows g and g+8 per 128-wide group. The contraction order inside a
//    group is permuted so that these 32 codes feed exactly the lane's A-fragment slots; the lane's
//    B fragment is the same 32 activations, re-paired with byte permutes. A dot product does not
//    depend on the order of its terms, so no weight re-layout is needed.
//  * int4 -> bf16 with the magic-exponent trick (codes are exact in bf16); the group's fp16 scale is
//    applied in fp32 to the group's partial sum (acc += s * partial), so weights are never rounded.
//  * Each lane streams its own 16-byte pieces into a private shared-memory ring with cp.async
//    (3 stages), keeping two groups of every warp in flight without holding them in registers.
// Gate/up mode computes both projections of the same 16 rows and writes h = silu(u) * v (bf16);
// down mode writes y (fp32) for the combine.
#include "kernels.cuh"

namespace strata {

constexpr int kWarpsPerCta = 8;
constexpr int kStages = 3;
constexpr int kTok = 8;  // token rows per work item (one n8 tile)

template <bool kGateUp>
__host__ __device__ constexpr int chunks_per_stage() {
  return (kGateUp ? 4 : 2) + 4;  // A pieces (2 rows x matrices) + 4 B pieces (64 bytes of x)
}

template <bool kGateUp>
size_t gemm_warp_smem() {
  return static_cast<size_t>(kWarpsPerCta) * kStages * chunks_per_stage<kGateUp>() * 32 * 16;
}

template <bool kGateUp>
__global__ void __launch_bounds__(256, 2) grouped_gemm_warp_kernel(GemmArgs a) {
  constexpr int NA = kGateUp ? 4 : 2;
  constexpr int NC = chunks_per_stage<kGateUp>();
  extern __shared__ uint4 smem_ring[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4* ring = smem_ring + warp * kStages * NC * 32;
  const int gq = lane >> 2, t4 = lane & 3;
  const int n_items = kGateUp ? a.hdr->n_items_gu : a.hdr->n_items_dn;
  const int nseg = a.hdr->nseg;
  const int total_warps = gridDim.x * kWarpsPerCta;
  const int slot = warp * gridDim.x + blockIdx.x;  // consecutive items land on different SMs
  const int ngroups = a.K / kGroup;
  const int mtiles = a.N / 16;
  const int64_t row_bytes = a.K / 2;
  const int64_t srow = a.K / kGroup;

  for (int item = slot; item < n_items; item += total_warps) {
    int lo = 0, hi = nseg - 1;  // segment s with seg_item[s] <= item < seg_item[s+1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.seg_item[mid] <= item) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int local = item - a.seg_item[s];
    const int chunk = local / mtiles, mt = local - chunk * mtiles;
    const int e = a.seg_expert[s];
    const int rbase = a.seg_row0[s] + chunk * kTok;
    const int nvalid = min(kTok, a.seg_rows[s] - chunk * kTok);

    const int64_t wrow = static_cast<int64_t>(e) * a.N + mt * 16 + gq;
    const uint8_t* A0 = a.codes0 + wrow * row_bytes + t4 * 16;
    const uint8_t* A1 = kGateUp ? a.codes1 + wrow * row_bytes + t4 * 16 : nullptr;
    const __half* S0 = a.scales0 + wrow * srow;
    const __half* S1 = kGateUp ? a.scales1 + wrow * srow : nullptr;
    const bool bvalid = gq < nvalid;
    int64_t src_row = 0;
    if (bvalid) src_row = kGateUp ? a.perm[rbase + gq] : (rbase + gq);
    const char* Bp = reinterpret_cast<const char*>(a.act + src_row * a.K + t4 * 32);

    auto issue = [&](int g) {
      uint4* st = ring + (g % kStages) * NC * 32 + lane;
      const int64_t off = static_cast<int64_t>(g) * 64;
      cp_async16(st + 0 * 32, A0 + off, true);
      cp_async16(st + 1 * 32, A0 + off + 8 * row_bytes, true);
      if (kGateUp) {
        cp_async16(st + 2 * 32, A1 + off, true);
        cp_async16(st + 3 * 32, A1 + off + 8 * row_bytes, true);
      }
      const char* b = Bp + static_cast<int64_t>(g) * 256;
#pragma unroll
      for (int c = 0; c < 4; ++c) cp_async16(st + (NA + c) * 32, b + c * 16, bvalid);
    };

    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int g = 0; g < kStages - 1; ++g) {
      if (g < ngroups) issue(g);
      cp_async_commit();
    }
    float s0l = __half2float(S0[0]), s0h = __half2float(S0[8 * srow]);
    float s1l = 0.f, s1h = 0.f;
    if (kGateUp) { s1l = __half2float(S1[0]); s1h = __half2float(S1[8 * srow]); }

    for (int g = 0; g < ngroups; ++g) {
      float n0l = 0.f, n0h = 0.f, n1l = 0.f, n1h = 0.f;  // next group's scales
      if (g + 1 < ngroups) {
        n0l = __half2float(S0[g + 1]);
        n0h = __half2float(S0[8 * srow + g + 1]);
        if (kGateUp) { n1l = __half2float(S1[g + 1]); n1h = __half2float(S1[8 * srow + g + 1]); }
      }
      cp_async_wait<kStages - 2>();
      __syncwarp();
      const uint4* st = ring + (g % kStages) * NC * 32 + lane;
      const uint4 a0l = st[0 * 32], a0h = st[1 * 32];
      uint4 a1l = make_uint4(0, 0, 0, 0), a1h = a1l;
      if (kGateUp) { a1l = st[2 * 32]; a1h = st[3 * 32]; }
      uint32_t X[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 b = st[(NA + c) * 32];
        X[4 * c + 0] = b.x; X[4 * c + 1] = b.y; X[4 * c + 2] = b.z; X[4 * c + 3] = b.w;
      }
      const uint32_t w0l[4] = {a0l.x, a0l.y, a0l.z, a0l.w}, w0h[4] = {a0h.x, a0h.y, a0h.z, a0h.w};
      const uint32_t w1l[4] = {a1l.x, a1l.y, a1l.z, a1l.w}, w1h[4] = {a1h.x, a1h.y, a1h.z, a1h.w};
      float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // B pairs: {x[8j], x[8j+4]}, {x[8j+1], x[8j+5]}, {x[8j+2], x[8j+6]}, {x[8j+3], x[8j+7]}
        const uint32_t b00 = prmt(X[4 * j], X[4 * j + 2], 0x5410);
        const uint32_t b01 = prmt(X[4 * j], X[4 * j + 2], 0x7632);
        const uint32_t b10 = prmt(X[4 * j + 1], X[4 * j + 3], 0x5410);
        const uint32_t b11 = prmt(X[4 * j + 1], X[4 * j + 3], 0x7632);
        {
          const uint32_t wl = w0l[j] ^ 0x88888888u, wh = w0h[j] ^ 0x88888888u;
          const uint32_t fa[4] = {int4pair_to_bf16x2(wl, 0), int4pair_to_bf16x2(wh, 0),
                                  int4pair_to_bf16x2(wl, 1), int4pair_to_bf16x2(wh, 1)};
          mma_bf16_16816(p0, fa, b00, b01, p0);
          const uint32_t fb[4] = {int4pair_to_bf16x2(wl, 2), int4pair_to_bf16x2(wh, 2),
                                  int4pair_to_bf16x2(wl, 3), int4pair_to_bf16x2(wh, 3)};
          mma_bf16_16816(p0, fb, b10, b11, p0);
        }
        if (kGateUp) {
          const uint32_t wl = w1l[j] ^ 0x88888888u, wh = w1h[j] ^ 0x88888888u;
          const uint32_t fa[4] = {int4pair_to_bf16x2(wl, 0), int4pair_to_bf16x2(wh, 0),
                                  int4pair_to_bf16x2(wl, 1), int4pair_to_bf16x2(wh, 1)};
          mma_bf16_16816(p1, fa, b00, b01, p1);
          const uint32_t fb[4] = {int4pair_to_bf16x2(wl, 2), int4pair_to_bf16x2(wh, 2),
                                  int4pair_to_bf16x2(wl, 3), int4pair_to_bf16x2(wh, 3)};
          mma_bf16_16816(p1, fb, b10, b11, p1);
        }
      }
      acc0[0] = fmaf(s0l, p0[0], acc0[0]); acc0[1] = fmaf(s0l, p0[1], acc0[1]);
      acc0[2] = fmaf(s0h, p0[2], acc0[2]); acc0[3] = fmaf(s0h, p0[3], acc0[3]);
      if (kGateUp) {
        acc1[0] = fmaf(s1l, p1[0], acc1[0]); acc1[1] = fmaf(s1l, p1[1], acc1[1]);
        acc1[2] = fmaf(s1h, p1[2], acc1[2]); acc1[3] = fmaf(s1h, p1[3], acc1[3]);
      }
      __syncwarp();
      if (g + kStages - 1 < ngroups) issue(g + kStages - 1);
      cp_async_commit();
      s0l = n0l; s0h = n0h; s1l = n1l; s1h = n1h;
    }
    cp_async_wait<0>();
    __syncwarp();

    // C fragment: c0,c1 -> weight row gq, token columns 2t4, 2t4+1; c2,c3 -> row gq+8
    const int n0 = mt * 16 + gq;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col = 2 * t4 + c;
      if (col >= nvalid) continue;
      const int64_t orow = rbase + col;
      if (kGateUp) {
        __nv_bfloat16* h = static_cast<__nv_bfloat16*>(a.out) + orow * a.N;
        h[n0] = __float2bfloat16_rn(silu_f(acc0[c]) * acc1[c]);
        h[n0 + 8] = __float2bfloat16_rn(silu_f(acc0[c + 2]) * acc1[c + 2]);
      } else {
        float* y = static_cast<float*>(a.out) + orow * a.N;
        y[n0] = acc0[c];
        y[n0 + 8] = acc0[c + 2];
      }
    }
  }
}

template <bool kGateUp>
cudaError_t launch_gemm_warp_t(const GemmArgs& a, int num_sms, cudaStream_t stream) {
  const size_t smem = gemm_warp_smem<kGateUp>();
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_warp_kernel<kGateUp>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  grouped_gemm_warp_kernel<kGateUp><<<num_sms * 2, kWarpsPerCta * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gemm_warp(const GemmArgs& a, bool gate_up, int num_sms, cudaStream_t stream) {
  return gate_up ? launch_gemm_warp_t<true>(a, num_sms, stream)
                 : launch_gemm_warp_t<false>(a, num_sms, stream);
}

}  // namespace strata
