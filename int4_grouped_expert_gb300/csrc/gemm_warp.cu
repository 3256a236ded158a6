// K4 (warp path): W4A16 grouped GEMM for segments with few rows — decode, where the layer is bound
// by streaming the activated experts' int4 weights from HBM. One launch covers every expert's
// group ("Strata" 3090 tuning, xdnf.cn/news/329730, §3.2: one grouped GEMM instead of one GEMM
// launch per expert); dequantization happens in registers ("Strata" architecture essay,
// dpshk.com/news/6309482, §3.2: decode is bandwidth-bound, so use wide vector loads and keep the
// small operands close).
//
// Work item = (8-row chunk of one expert's rows, two 16-row weight tiles[, contraction split]).
// Gate/up: the two tiles are the gate and up rows of the same 16 outputs; down: two consecutive
// 16-row tiles. Warps pull items from a device counter and read the chunk from a flat list.
// A warp computes its item with mma.sync m16n8k16 (bf16 in, fp32 accumulate) and swapped
// operands: weight rows are the A operand, the (up to 8) tokens the B operand.
//  * Codes are read in their canonical row-major layout. Lane (g = lane/4, t = lane%4) takes 16
//    bytes = 32 codes of rows g and g+8 per 128-wide group, and the contraction order inside the
//    group is permuted so that they feed exactly the lane's A-fragment slots. The activations are
//    stored with every 8-wide chunk in (0,4,1,5,2,6,3,7) order (x by the router, h by the gate/up
//    epilogue), which is exactly the B-fragment pairing, so B needs no byte permutes. A dot
//    product does not depend on the order of its terms, so no weight re-layout is needed.
//  * int4 -> bf16 in one LOP3 per code pair: flipping each nibble's sign bit and OR-ing it into
//    the low mantissa of bf16 128 yields q + 136 exactly. The +136 is removed after the group's
//    MMAs with a correction MMA (A = 136 everywhere, same B) shared by both tiles, and the group's
//    fp16 scale is applied in fp32: acc += s * (partial - correction). Weights are never rounded.
//  * Every lane streams its own 16-byte pieces (weights, and activations for lanes that carry a
//    token) into a private cp.async ring 6 groups deep; scales come 4 groups ahead through
//    registers. The loop body only reads shared memory and computes.
//  * Tiny batches split the gate/up contraction; the last split to arrive (device counter) sums
//    the partials in split order and applies the epilogue, so results stay deterministic.
// Gate/up writes h = silu(u) * v (bf16); down writes y (fp32) for the combine.
#include "kernels.cuh"

namespace strata {

#ifndef STRATA_WARP_WARPS
#define STRATA_WARP_WARPS 12
#endif
#ifndef STRATA_WARP_STAGES
#define STRATA_WARP_STAGES 4
#endif
#ifndef STRATA_WARP_MULHI_SHIFT
#define STRATA_WARP_MULHI_SHIFT 0
#endif
constexpr int kWarpsPerCta = STRATA_WARP_WARPS;  // one CTA per SM
constexpr int kStages = STRATA_WARP_STAGES;      // groups in the cp.async ring of every warp
constexpr int kNC = 8;      // 16-byte pieces per lane per group: 4 weight + 4 activation
constexpr int kSD = 4;      // scale prefetch distance (groups)

size_t gemm_warp_smem() { return static_cast<size_t>(kWarpsPerCta) * kStages * kNC * 32 * 16; }

// pair i of an 8-code word (two's complement nibbles) as bf16x2 {q_i + 136, q_{i+4} + 136}.
// v = w >> 4i comes in precomputed (see shifted()).
__device__ __forceinline__ uint32_t codes_to_bf16_biased(uint32_t v) {
  uint32_t d;
  // d = mask ? (v ^ c) : c, mask = 0x000F000F, c = 0x43084308: flips the nibble sign bits and
  // puts the exponent of 128 around them
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(v), "n"(0x000F000F), "n"(0x43084308));
  return d;
}

// w >> 4, w >> 8, w >> 12 as high halves of 32x32 products (the multipliers 2^28, 2^24, 2^20 are
// kernel arguments, so the compiler keeps the integer multiply): the shifts run on the FMA pipe
// and leave the ALU pipe to the LOP3s.
struct Shifts {
  uint32_t m4, m8, m12;
};
__device__ __forceinline__ void shifted(uint32_t w, const Shifts& k, uint32_t (&v)[4]) {
  v[0] = w;
#if STRATA_WARP_MULHI_SHIFT
  v[1] = __umulhi(w, k.m4);
  v[2] = __umulhi(w, k.m8);
  v[3] = __umulhi(w, k.m12);
#else
  v[1] = w >> 4;
  v[2] = w >> 8;
  v[3] = w >> 12;
#endif
}

// mode: true = gate/up (tiles are gate and up of the same rows), false = down (two row tiles)
template <bool kGateUp>
__global__ void __launch_bounds__(kWarpsPerCta * 32, 1) grouped_gemm_warp_kernel(GemmArgs a, Shifts sh) {
  extern __shared__ uint4 smem_ring[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4* ring = smem_ring + warp * kStages * kNC * 32 + lane;
  // Gate/up reads the router's work lists: wait for it. Down reads h from gate/up, but its work
  // lists come from the router (complete before gate/up started), so it streams its first item's
  // weights before waiting (below).
  if (kGateUp) griddep_wait();
  griddep_launch();
  bool first = true;
  const int gq = lane >> 2, t4 = lane & 3;
  int* const next_ctr = kGateUp ? &a.hdr->next_gu : &a.hdr->next_dn;
  const int n_items = kGateUp ? a.hdr->n_items_gu : a.hdr->n_items_dn;
  const int nchunks = a.hdr->n_chunks;
  const int KS = kGateUp ? a.ksplit : 1;
  const int ngroups = a.K / kGroup;
  const int mtiles = kGateUp ? a.N / 16 : a.N / 32;
  const int64_t row_bytes = a.K / 2;
  const int64_t srow = a.K / kGroup;
  const uint32_t a136[4] = {0x43084308u, 0x43084308u, 0x43084308u, 0x43084308u};

  int item = 0;
  if (lane == 0) item = atomicAdd(next_ctr, 1);
  item = __shfl_sync(0xffffffffu, item, 0);
  int4 ch = make_int4(0, 0, 0, 0);
  if (item < n_items) ch = __ldg(a.chunk_list + item % nchunks);
  if (!kGateUp && item >= n_items) griddep_wait();  // no work: still order the exit
  while (item < n_items) {
    int nxt = 0;
    if (lane == 0) nxt = atomicAdd(next_ctr, 1);  // next item, fetched while this one runs

    // item -> (contraction split, row tile, chunk): chunk fastest, so consecutive items stream
    // different experts' rows
    const int cidx = item % nchunks;
    const int rest = item / nchunks;
    const int mt = rest % mtiles;
    const int ks = rest / mtiles;
    const int e = ch.x;
    const int rbase = ch.y;
    const int nvalid = ch.z;
    const int gbeg = (ks * ngroups) / KS, gend = ((ks + 1) * ngroups) / KS;

    // A tiles: rows r0 and r1 (16 rows each) of matrices m0 / m1
    const int64_t rowA = static_cast<int64_t>(e) * a.N + (kGateUp ? mt * 16 : mt * 32) + gq;
    const int64_t rowB = kGateUp ? rowA : rowA + 16;
    const uint8_t* A0 = a.codes0 + rowA * row_bytes + t4 * 16;
    const uint8_t* A1 = (kGateUp ? a.codes1 : a.codes0) + rowB * row_bytes + t4 * 16;
    const __half* S0 = a.scales0 + rowA * srow;
    const __half* S1 = (kGateUp ? a.scales1 : a.scales0) + rowB * srow;
    const bool bvalid = gq < nvalid;
    int64_t src_row = 0;
    if (bvalid) src_row = a.perm ? a.perm[rbase + gq] : (rbase + gq);
    const char* Bp = reinterpret_cast<const char*>(a.act + src_row * a.K + t4 * 32);

    auto issue_a = [&](int g, int slot) {
      uint4* st = ring + slot * kNC * 32;
      const int64_t off = static_cast<int64_t>(g) * 64;
      cp_async16(st + 0 * 32, A0 + off, true);
      cp_async16(st + 1 * 32, A0 + off + 8 * row_bytes, true);
      cp_async16(st + 2 * 32, A1 + off, true);
      cp_async16(st + 3 * 32, A1 + off + 8 * row_bytes, true);
    };
    auto issue_b = [&](int g, int slot) {
      uint4* st = ring + slot * kNC * 32;
      const char* b = Bp + static_cast<int64_t>(g) * 256;
#pragma unroll
      for (int c = 0; c < 4; ++c) cp_async16(st + (4 + c) * 32, b + c * 16, bvalid);
    };
    auto issue = [&](int g, int slot) {
      issue_a(g, slot);
      issue_b(g, slot);
    };
    // scales of groups g .. g+kSD-1 in fixed slots, kept as raw fp16 bits until used (converting
    // on load would make every load complete at once): [i] = rows gq, gq+8 of tile 0, then tile 1
    uint32_t sc[kSD][2];
    auto load_sc = [&](int g, uint32_t (&d)[2]) {
      if (g < gend) {
        const unsigned short a0 = __ldg(reinterpret_cast<const unsigned short*>(S0) + g);
        const unsigned short a1 = __ldg(reinterpret_cast<const unsigned short*>(S0) + 8 * srow + g);
        const unsigned short b0 = __ldg(reinterpret_cast<const unsigned short*>(S1) + g);
        const unsigned short b1 = __ldg(reinterpret_cast<const unsigned short*>(S1) + 8 * srow + g);
        d[0] = static_cast<uint32_t>(a0) | (static_cast<uint32_t>(a1) << 16);
        d[1] = static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 16);
      }
    };
#pragma unroll
    for (int i = 0; i < kSD; ++i) load_sc(gbeg + i, sc[i]);
    if (!kGateUp && first) {
      // down's first item: weights first, then wait for gate/up's h, then the activations
#pragma unroll
      for (int i = 0; i < kStages - 1; ++i) {
        if (gbeg + i < gend) issue_a(gbeg + i, i);
        cp_async_commit();
      }
      griddep_wait();
#pragma unroll
      for (int i = 0; i < kStages - 1; ++i)
        if (gbeg + i < gend) issue_b(gbeg + i, i);
      cp_async_commit();
      cp_async_wait<0>();
    } else {
#pragma unroll
      for (int i = 0; i < kStages - 1; ++i) {
        if (gbeg + i < gend) issue(gbeg + i, i);
        cp_async_commit();
      }
    }
    first = false;
    int rd = 0, wr = kStages - 1;  // ring slots of the group read now / the group issued next
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    int4 ch_next = ch;
    bool fetched = false;
    // kSD groups per outer step, fully unrolled, so scale slot u is a fixed register set that is
    // refilled for group g + kSD right after group g used it (kSD groups of latency to hide)
    for (int g0 = gbeg; g0 < gend; g0 += kSD) {
#pragma unroll
      for (int u = 0; u < kSD; ++u) {
        const int g = g0 + u;
        if (g >= gend) break;
        cp_async_wait<kStages - 2>();
        __syncwarp();
        const uint4* st = ring + rd * kNC * 32;
        const uint4 a0l = st[0 * 32], a0h = st[1 * 32], a1l = st[2 * 32], a1h = st[3 * 32];
        uint32_t X[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 b = st[(4 + c) * 32];
          X[4 * c] = b.x; X[4 * c + 1] = b.y; X[4 * c + 2] = b.z; X[4 * c + 3] = b.w;
        }
        const uint32_t w0l[4] = {a0l.x, a0l.y, a0l.z, a0l.w}, w0h[4] = {a0h.x, a0h.y, a0h.z, a0h.w};
        const uint32_t w1l[4] = {a1l.x, a1l.y, a1l.z, a1l.w}, w1h[4] = {a1h.x, a1h.y, a1h.z, a1h.w};
        // two accumulator sets (even / odd j) halve the MMA dependency chains
        float p0[2][4] = {}, p1[2][4] = {}, cr[2][4] = {};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int h = j & 1;
          // activations are stored pair-interleaved: X[4j+m] = {x[8j+m], x[8j+m+4]}
          const uint32_t b00 = X[4 * j], b01 = X[4 * j + 1], b10 = X[4 * j + 2], b11 = X[4 * j + 3];
          mma_bf16_16816(cr[h], a136, b00, b01, cr[h]);
          mma_bf16_16816(cr[h], a136, b10, b11, cr[h]);
          uint32_t vl[4], vh[4];
          shifted(w0l[j], sh, vl);
          shifted(w0h[j], sh, vh);
          {
            const uint32_t fa[4] = {codes_to_bf16_biased(vl[0]), codes_to_bf16_biased(vh[0]),
                                    codes_to_bf16_biased(vl[1]), codes_to_bf16_biased(vh[1])};
            mma_bf16_16816(p0[h], fa, b00, b01, p0[h]);
            const uint32_t fb[4] = {codes_to_bf16_biased(vl[2]), codes_to_bf16_biased(vh[2]),
                                    codes_to_bf16_biased(vl[3]), codes_to_bf16_biased(vh[3])};
            mma_bf16_16816(p0[h], fb, b10, b11, p0[h]);
          }
          shifted(w1l[j], sh, vl);
          shifted(w1h[j], sh, vh);
          {
            const uint32_t fa[4] = {codes_to_bf16_biased(vl[0]), codes_to_bf16_biased(vh[0]),
                                    codes_to_bf16_biased(vl[1]), codes_to_bf16_biased(vh[1])};
            mma_bf16_16816(p1[h], fa, b00, b01, p1[h]);
            const uint32_t fb[4] = {codes_to_bf16_biased(vl[2]), codes_to_bf16_biased(vh[2]),
                                    codes_to_bf16_biased(vl[3]), codes_to_bf16_biased(vh[3])};
            mma_bf16_16816(p1[h], fb, b10, b11, p1[h]);
          }
        }
        float q0[4], q1[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          q0[c] = (p0[0][c] - cr[0][c]) + (p0[1][c] - cr[1][c]);
          q1[c] = (p1[0][c] - cr[0][c]) + (p1[1][c] - cr[1][c]);
        }
        const float2 s0 = __half22float2(*reinterpret_cast<const __half2*>(&sc[u][0]));
        const float2 s1 = __half22float2(*reinterpret_cast<const __half2*>(&sc[u][1]));
        acc0[0] = fmaf(s0.x, q0[0], acc0[0]); acc0[1] = fmaf(s0.x, q0[1], acc0[1]);
        acc0[2] = fmaf(s0.y, q0[2], acc0[2]); acc0[3] = fmaf(s0.y, q0[3], acc0[3]);
        acc1[0] = fmaf(s1.x, q1[0], acc1[0]); acc1[1] = fmaf(s1.x, q1[1], acc1[1]);
        acc1[2] = fmaf(s1.y, q1[2], acc1[2]); acc1[3] = fmaf(s1.y, q1[3], acc1[3]);
        load_sc(g + kSD, sc[u]);
        __syncwarp();
        if (g + kStages - 1 < gend) issue(g + kStages - 1, wr);
        cp_async_commit();
        rd = (rd + 1 == kStages) ? 0 : rd + 1;
        wr = (wr + 1 == kStages) ? 0 : wr + 1;
        if (!fetched) {  // the next item's chunk entry, while this item streams
          fetched = true;
          const int n = __shfl_sync(0xffffffffu, nxt, 0);
          if (n < n_items) ch_next = __ldg(a.chunk_list + n % nchunks);
        }
      }
    }
    if (!fetched) {  // empty contraction split
      const int n = __shfl_sync(0xffffffffu, nxt, 0);
      if (n < n_items) ch_next = __ldg(a.chunk_list + n % nchunks);
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
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col = 2 * t4 + c;
        if (col >= nvalid) continue;
        const int64_t orow = rbase + col;
        if (kGateUp) {
          // h columns are stored pair-interleaved inside every 8 (the down GEMM's B order)
          const int n0 = mt * 16 + (gq < 4 ? 2 * gq : 2 * gq - 7);
          __nv_bfloat16* h = static_cast<__nv_bfloat16*>(a.out) + orow * a.N;
          h[n0] = __float2bfloat16_rn(silu_f(acc0[c]) * acc1[c]);
          h[n0 + 8] = __float2bfloat16_rn(silu_f(acc0[c + 2]) * acc1[c + 2]);
        } else {
          const int n0 = mt * 32 + gq;
          float* y = static_cast<float*>(a.out) + orow * a.N;
          y[n0] = acc0[c];
          y[n0 + 8] = acc0[c + 2];
          y[n0 + 16] = acc1[c];
          y[n0 + 24] = acc1[c + 2];
        }
      }
    }
    item = __shfl_sync(0xffffffffu, nxt, 0);
    ch = ch_next;
  }
}

template <bool kGateUp>
cudaError_t launch_gemm_warp_t(const GemmArgs& a, int num_sms, cudaStream_t stream) {
  const size_t smem = gemm_warp_smem();
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_warp_kernel<kGateUp>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const Shifts sh{1u << 28, 1u << 24, 1u << 20};
  return launch_kernel(grouped_gemm_warp_kernel<kGateUp>, dim3(num_sms), dim3(kWarpsPerCta * 32),
                       smem, stream, true, a, sh);
}

cudaError_t launch_gemm_warp(const GemmArgs& a, bool gate_up, int num_sms, cudaStream_t stream) {
  return gate_up ? launch_gemm_warp_t<true>(a, num_sms, stream)
                 : launch_gemm_warp_t<false>(a, num_sms, stream);
}

// contraction splits of the gate/up warp path for a batch of T tokens: enough items for ~2 per warp
int warp_ksplit(int64_t T, int E, int k, int shared, int64_t I, int64_t H) {
  const int64_t segs = (T * k < E ? T * k : E) + shared;
  const int64_t items = segs * (I / 16);
  const int64_t want = 2 * 152 * kWarpsPerCta;
  int ks = 4;
  if (items >= want) ks = 1;
  else if (2 * items >= want) ks = 2;
  const int64_t groups = H / kGroup;  // every split keeps at least one 128-wide group
  while (ks > 1 && ks > groups) ks /= 2;
  return ks;
}

}  // namespace strata
