// K4 (warp path): W4A16 grouped GEMM for segments with few rows — decode, where the layer is bound
// by streaming the activated experts' int4 weights from HBM. One launch covers every expert's
// group ("Strata" 3090 tuning, xdnf.cn/news/329730, §3.2: one grouped GEMM instead of one GEMM
// launch per expert); dequantization happens in registers ("Strata" architecture essay,
// dpshk.com/news/6309482, §3.2: decode is bandwidth-bound, so use wide vector loads and keep the
// small operands close).
//
// Work item = (8-row chunk of one expert's rows, 16 weight rows[, contraction split]); warps pull
// items from a device counter and read the chunk from a flat list (no search). A warp computes its item with mma.sync m16n8k16 (bf16 in, fp32
// accumulate) and swapped operands: the 16 weight rows are the A operand, the tokens the 8-wide B.
//  * Codes are read in their canonical row-major layout. Lane (g = lane/4, t = lane%4) takes 16
//    bytes = 32 codes of rows g and g+8 per 128-wide group, and the contraction order inside the
//    group is permuted so that they feed exactly the lane's A-fragment slots; the lane's B fragment
//    is the same 32 activations, re-paired with byte permutes. A dot product does not depend on
//    the order of its terms, so no weight re-layout is needed.
//  * int4 -> bf16 in one LOP3 per code pair: flipping each nibble's sign bit and OR-ing it into
//    the low mantissa of bf16 128 yields q + 136 exactly. The +136 is removed after the group's
//    MMAs with a correction MMA (A = 136 everywhere, same B) shared by gate and up, and the
//    group's fp16 scale is applied in fp32: acc += s * (partial - correction). Weights are
//    never rounded.
//  * Only the weight stream goes through shared memory: each lane copies its own 16-byte pieces
//    into a private cp.async ring (6 groups deep for gate/up, 10 for down). Activations (a few
//    rows, L2-resident) are loaded into registers one group ahead.
//  * Tiny batches split the gate/up contraction; the last split to arrive (device counter) sums
//    the partials in split order and applies the epilogue, so results stay deterministic.
// Gate/up mode computes both projections of the same 16 rows and writes h = silu(u) * v (bf16);
// down mode writes y (fp32) for the combine.
#include "kernels.cuh"

namespace strata {

constexpr int kWarpsPerCta = 8;
constexpr int kTok = 8;  // token rows per work item (one n8 tile)

template <bool kGateUp>
struct WarpCfg {
  static constexpr int NA = kGateUp ? 4 : 2;     // 16-byte A pieces per lane per group
  static constexpr int S = kGateUp ? 6 : 10;     // groups in flight per warp
};

template <bool kGateUp>
size_t gemm_warp_smem() {
  return static_cast<size_t>(kWarpsPerCta) * WarpCfg<kGateUp>::S * WarpCfg<kGateUp>::NA * 32 * 16;
}

// pair i of an 8-code word (two's complement nibbles) as bf16x2 {q_i + 136, q_{i+4} + 136}
__device__ __forceinline__ uint32_t codes_to_bf16_biased(uint32_t w, int i) {
  const uint32_t v = w >> (4 * i);
  uint32_t d;
  // d = mask ? (v ^ c) : c, mask = 0x000F000F, c = 0x43084308: flips the nibble sign bits and
  // puts the exponent of 128 around them
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(v), "n"(0x000F000F), "n"(0x43084308));
  return d;
}

__device__ __forceinline__ uint4 ldg16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

template <bool kGateUp>
__global__ void __launch_bounds__(256, 2) grouped_gemm_warp_kernel(GemmArgs a) {
  constexpr int NA = WarpCfg<kGateUp>::NA;
  constexpr int S = WarpCfg<kGateUp>::S;
  extern __shared__ uint4 smem_ring[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4* ring = smem_ring + warp * S * NA * 32 + lane;
  const int gq = lane >> 2, t4 = lane & 3;
  int* const next_ctr = kGateUp ? &a.hdr->next_gu : &a.hdr->next_dn;
  const int n_items = kGateUp ? a.hdr->n_items_gu : a.hdr->n_items_dn;
  const int nchunks = a.hdr->n_chunks;
  const int KS = kGateUp ? a.ksplit : 1;
  const int ngroups = a.K / kGroup;
  const int mtiles = a.N / 16;
  const int64_t row_bytes = a.K / 2;
  const int64_t srow = a.K / kGroup;
  const uint32_t a136[4] = {0x43084308u, 0x43084308u, 0x43084308u, 0x43084308u};

  int item = 0;
  if (lane == 0) item = atomicAdd(next_ctr, 1);
  item = __shfl_sync(0xffffffffu, item, 0);
  while (item < n_items) {
    int nxt = 0;
    if (lane == 0) nxt = atomicAdd(next_ctr, 1);  // next item, fetched while this one runs

    // item -> (contraction split, row tile, chunk): chunk fastest, so consecutive items stream
    // different experts' rows
    const int cidx = item % nchunks;
    const int rest = item / nchunks;
    const int mt = rest % mtiles;
    const int ks = rest / mtiles;
    const int4 ch = __ldg(a.chunk_list + cidx);
    const int e = ch.x;
    const int rbase = ch.y;
    const int nvalid = ch.z;
    const int gbeg = (ks * ngroups) / KS, gend = ((ks + 1) * ngroups) / KS;

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
      uint4* st = ring + ((g - gbeg) % S) * NA * 32;
      const int64_t off = static_cast<int64_t>(g) * 64;
      cp_async16(st + 0 * 32, A0 + off, true);
      cp_async16(st + 1 * 32, A0 + off + 8 * row_bytes, true);
      if (kGateUp) {
        cp_async16(st + 2 * 32, A1 + off, true);
        cp_async16(st + 3 * 32, A1 + off + 8 * row_bytes, true);
      }
    };
    auto load_b = [&](int g, uint32_t (&X)[16]) {
      if (bvalid) {
        const char* b = Bp + static_cast<int64_t>(g) * 256;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = ldg16(b + c * 16);
          X[4 * c] = v.x; X[4 * c + 1] = v.y; X[4 * c + 2] = v.z; X[4 * c + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) X[c] = 0u;
      }
    };

#pragma unroll
    for (int i = 0; i < S - 1; ++i) {
      if (gbeg + i < gend) issue(gbeg + i);
      cp_async_commit();
    }
    uint32_t X[16];
    load_b(gbeg, X);
    float s0l = __half2float(S0[gbeg]), s0h = __half2float(S0[8 * srow + gbeg]);
    float s1l = 0.f, s1h = 0.f;
    if (kGateUp) { s1l = __half2float(S1[gbeg]); s1h = __half2float(S1[8 * srow + gbeg]); }
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};

    for (int g = gbeg; g < gend; ++g) {
      uint32_t Xn[16];
      float n0l = 0.f, n0h = 0.f, n1l = 0.f, n1h = 0.f;
      if (g + 1 < gend) {
        load_b(g + 1, Xn);
        n0l = __half2float(S0[g + 1]);
        n0h = __half2float(S0[8 * srow + g + 1]);
        if (kGateUp) { n1l = __half2float(S1[g + 1]); n1h = __half2float(S1[8 * srow + g + 1]); }
      }
      cp_async_wait<S - 2>();
      __syncwarp();
      const uint4* st = ring + ((g - gbeg) % S) * NA * 32;
      const uint4 a0l = st[0 * 32], a0h = st[1 * 32];
      uint4 a1l = make_uint4(0, 0, 0, 0), a1h = a1l;
      if (kGateUp) { a1l = st[2 * 32]; a1h = st[3 * 32]; }
      const uint32_t w0l[4] = {a0l.x, a0l.y, a0l.z, a0l.w}, w0h[4] = {a0h.x, a0h.y, a0h.z, a0h.w};
      const uint32_t w1l[4] = {a1l.x, a1l.y, a1l.z, a1l.w}, w1h[4] = {a1h.x, a1h.y, a1h.z, a1h.w};
      float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f}, cr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // B pairs: {x[8j], x[8j+4]}, {x[8j+1], x[8j+5]}, {x[8j+2], x[8j+6]}, {x[8j+3], x[8j+7]}
        const uint32_t b00 = prmt(X[4 * j], X[4 * j + 2], 0x5410);
        const uint32_t b01 = prmt(X[4 * j], X[4 * j + 2], 0x7632);
        const uint32_t b10 = prmt(X[4 * j + 1], X[4 * j + 3], 0x5410);
        const uint32_t b11 = prmt(X[4 * j + 1], X[4 * j + 3], 0x7632);
        mma_bf16_16816(cr, a136, b00, b01, cr);
        mma_bf16_16816(cr, a136, b10, b11, cr);
        {
          const uint32_t fa[4] = {codes_to_bf16_biased(w0l[j], 0), codes_to_bf16_biased(w0h[j], 0),
                                  codes_to_bf16_biased(w0l[j], 1), codes_to_bf16_biased(w0h[j], 1)};
          mma_bf16_16816(p0, fa, b00, b01, p0);
          const uint32_t fb[4] = {codes_to_bf16_biased(w0l[j], 2), codes_to_bf16_biased(w0h[j], 2),
                                  codes_to_bf16_biased(w0l[j], 3), codes_to_bf16_biased(w0h[j], 3)};
          mma_bf16_16816(p0, fb, b10, b11, p0);
        }
        if (kGateUp) {
          const uint32_t fa[4] = {codes_to_bf16_biased(w1l[j], 0), codes_to_bf16_biased(w1h[j], 0),
                                  codes_to_bf16_biased(w1l[j], 1), codes_to_bf16_biased(w1h[j], 1)};
          mma_bf16_16816(p1, fa, b00, b01, p1);
          const uint32_t fb[4] = {codes_to_bf16_biased(w1l[j], 2), codes_to_bf16_biased(w1h[j], 2),
                                  codes_to_bf16_biased(w1l[j], 3), codes_to_bf16_biased(w1h[j], 3)};
          mma_bf16_16816(p1, fb, b10, b11, p1);
        }
      }
      acc0[0] = fmaf(s0l, p0[0] - cr[0], acc0[0]); acc0[1] = fmaf(s0l, p0[1] - cr[1], acc0[1]);
      acc0[2] = fmaf(s0h, p0[2] - cr[2], acc0[2]); acc0[3] = fmaf(s0h, p0[3] - cr[3], acc0[3]);
      if (kGateUp) {
        acc1[0] = fmaf(s1l, p1[0] - cr[0], acc1[0]); acc1[1] = fmaf(s1l, p1[1] - cr[1], acc1[1]);
        acc1[2] = fmaf(s1h, p1[2] - cr[2], acc1[2]); acc1[3] = fmaf(s1h, p1[3] - cr[3], acc1[3]);
      }
      __syncwarp();
      if (g + S - 1 < gend) issue(g + S - 1);
      cp_async_commit();
#pragma unroll
      for (int c = 0; c < 16; ++c) X[c] = Xn[c];
      s0l = n0l; s0h = n0h; s1l = n1l; s1h = n1h;
    }
    cp_async_wait<0>();
    __syncwarp();

    bool write = true;
    if (kGateUp && KS > 1) {
      // split-K: publish this split's partial sums; the last split to arrive reduces them
      const int tile = cidx * mtiles + mt;
      float* part = a.split_part + (static_cast<int64_t>(tile) * KS + ks) * 256 + lane * 8;
      reinterpret_cast<float4*>(part)[0] = make_float4(acc0[0], acc0[1], acc0[2], acc0[3]);
      reinterpret_cast<float4*>(part)[1] = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = (atomicAdd(a.split_cnt + tile, 1) == KS - 1);
      last = __shfl_sync(0xffffffffu, last, 0);
      write = last != 0;
      if (last) {
        __threadfence();
        const float* base = a.split_part + static_cast<int64_t>(tile) * KS * 256 + lane * 8;
#pragma unroll
        for (int c = 0; c < 4; ++c) { acc0[c] = 0.f; acc1[c] = 0.f; }
        for (int q = 0; q < KS; ++q) {  // split order: deterministic
          const float4 u = __ldcg(reinterpret_cast<const float4*>(base + q * 256));
          const float4 v = __ldcg(reinterpret_cast<const float4*>(base + q * 256) + 1);
          acc0[0] += u.x; acc0[1] += u.y; acc0[2] += u.z; acc0[3] += u.w;
          acc1[0] += v.x; acc1[1] += v.y; acc1[2] += v.z; acc1[3] += v.w;
        }
      }
    }
    if (write) {
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
    item = __shfl_sync(0xffffffffu, nxt, 0);
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

// contraction splits of the gate/up warp path for a batch of T tokens: enough items for ~2 per warp
int warp_ksplit(int64_t T, int E, int k, int shared, int64_t I) {
  const int64_t segs = (T * k < E ? T * k : E) + shared;
  const int64_t items = segs * (I / 16);
  const int64_t want = 2 * 152 * 2 * kWarpsPerCta;
  if (items >= want) return 1;
  if (2 * items >= want) return 2;
  return 4;
}

}  // namespace strata
