// K4 (tensor-core path): W4A16 grouped GEMM on tcgen05 for segments with many rows (prefill),
// where the expert FFN is a dense contraction. One persistent launch covers every expert's group
// ("Strata" 3090 tuning, xdnf.cn/news/329730, §3.2: one grouped GEMM for all experts); the int4
// weights are dequantized on chip ("Strata" MoE tuning notes, lpnh.cn/news/2730718, §2.1 format:
// 128 codes share one fp16 scale).
//
// Tile = (segment, 128 weight rows, up to kN token rows), contraction in 64-wide stages.
//   warp 0       TMA producer: the stage's token rows (f16, 128-byte swizzle) -> shared memory
//   warp 1       MMA issuer: one thread issues tcgen05.mma (M=128, N=rows, K=16) into TMEM
//   warp 2       owns the TMEM allocation
//   warp 3       small tiles only: TMA producer of the int4 code tiles (a deep ring of stages)
//   warps 4..    dequant producers (16 warps for 256-row gate/up tiles, 8 otherwise): int4
//                codes -> f16(q*s) written in the same swizzled K-major layout (the A operand)
//   last 4 warps epilogue: TMEM -> registers -> global
// Two tile widths: kN = 256 token rows for segments with many rows (the dequant warps load their
// codes from global memory themselves, four stages ahead in registers), and kN = 64 for batches
// with few rows per expert. There the shared memory the wide B tiles would take holds a ring of
// code tiles filled by TMA (slots of four stages: 128-byte rows), so that enough weight bytes are
// in flight to stream HBM while each dequantized tile serves only a few dozen tokens.
// D[weight row][token] accumulates in TMEM: gate/up in one 512-column buffer (gate, then up);
// down in two 256-column buffers, so its MMAs for the next tile run while the epilogue drains
// this one. While the epilogue runs, the dequant warps already fill the next tile's stages.
// Gate/up writes h = silu(gate) * up as f16; down writes y in fp32 for the combine.
//
// Contraction order: inside every 8-wide chunk the K order is (0,4,1,5,2,6,3,7). That is the
// order in which one LOP3 per pair unpacks the codes, so the activations are stored in it too (by
// the gather kernel for x, by the gate/up epilogue for h); a dot product is order-independent.
//
// Operands are f16 (tcgen05.mma kind::f16 with f16 A and B): the weight is w = f16(q * s), the
// exact code times the fp16 scale rounded once (2^-11 relative); x (gathered by the row kernel)
// and h (written by the gate/up epilogue) are f16, exact from bf16 within the f16 range and
// saturated at +-65504 outside it.
//
// Every mbarrier wait is bounded in time; on time-out the kernel sets STRATA_DEV_TIMEOUT, every
// role leaves its loop, in-flight copies and MMAs are drained (bounded) and TMEM is freed.
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace strata {

constexpr int kTcBM = 128;       // weight rows per tile (MMA M)
constexpr int kTcBK = 64;        // contraction per stage: one 128-byte swizzle row of f16


#ifndef STRATA_TC_SMALL_STAGES_GU
#define STRATA_TC_SMALL_STAGES_GU 3
#endif
#ifndef STRATA_TC_SMALL_RING_GU
#define STRATA_TC_SMALL_RING_GU 3
#endif
#ifndef STRATA_TC_SMALL_STAGES_DN
#define STRATA_TC_SMALL_STAGES_DN 4
#endif
#ifndef STRATA_TC_SMALL_RING_DN
#define STRATA_TC_SMALL_RING_DN 4
#endif
template <bool kGateUp, int kN, int kBits = 4>
struct TcCfg {
  static constexpr bool RING = kN <= 64;               // code tiles through the TMA ring
  static constexpr int STAGES = RING ? (kGateUp ? STRATA_TC_SMALL_STAGES_GU : STRATA_TC_SMALL_STAGES_DN)
                                     : (kGateUp ? 3 : 4);
  static constexpr int A_BYTES = kTcBM * kTcBK * 2;    // 16 KB per weight matrix
  static constexpr int B_BYTES = kN * kTcBK * 2;       // 32 KB (kN = 256) or 8 KB (64)
  // TMA box of token rows x 64 columns: the whole tile for 64-row tiles, else 32 rows, so that a
  // stage loads only the boxes its MMAs read (the B tile's shared-memory writes are part of the
  // per-stage traffic that bounds these kernels)
  static constexpr int BOX_ROWS = kN < 128 ? kN : 32;
  static constexpr int BOX_BYTES = BOX_ROWS * kTcBK * 2;
  static constexpr int NMAT = kGateUp ? 2 : 1;
  static constexpr int STAGE_BYTES = NMAT * A_BYTES + B_BYTES;
  // dequant producer warps: 16 for the 256-row gate/up tiles, whose stage conversion (two
  // matrices) is the kernel's critical chain; 8 elsewhere (more were slower there)
  static constexpr int DQW = (kGateUp && !RING) ? 16 : 8;
  static constexpr int THREADS = (4 + DQW + 4) * 32;  // + 4 role warps + 4 epilogue warps
  // ring slot: the codes of SLOT_K consecutive stages (128 bytes of every weight row, one TMA box
  // of 128 rows per matrix, 128-byte swizzle): four stages of 4-bit codes or two of 8-bit ones
  static constexpr int STAGE_CODE_BYTES = kTcBK * kBits / 8;  // bytes of one row per stage
  static constexpr int SLOT_K = 128 / STAGE_CODE_BYTES;
  static constexpr int CODE_BYTES = NMAT * kTcBM * 128;
  static constexpr int RING_STAGES = RING ? (kGateUp ? STRATA_TC_SMALL_RING_GU : STRATA_TC_SMALL_RING_DN) : 0;
  static constexpr uint32_t ACC_COLS = NMAT * kN;        // one accumulator buffer
  static constexpr int NBUF = (kGateUp && !RING) ? 1 : 2;  // accumulator buffers (<= 512 columns)
  static constexpr uint32_t TMEM_COLS = NBUF * ACC_COLS;
  static constexpr size_t SMEM =
      static_cast<size_t>(STAGES) * STAGE_BYTES + static_cast<size_t>(RING_STAGES) * CODE_BYTES +
      1024 + 512;
};

struct TcTile {
  int e, mt, row0, nvalid, nmma;
};

template <int kN>
__device__ __forceinline__ bool tc_decode(const TcArgs& a, int item, int nseg, int mtiles,
                                          TcTile& t) {
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.seg_item[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int local = item - a.seg_item[lo];
  const int chunk = local / mtiles;
  t.mt = local - chunk * mtiles;
  t.e = a.seg_expert[lo];
  t.row0 = a.seg_row0[lo] + chunk * kN;
  t.nvalid = min(kN, a.seg_rows[lo] - chunk * kN);
  t.nmma = (t.nvalid + 15) & ~15;
  return true;
}

// f16x2 {q_i, q_{i+4}} of an 8-code word (two's complement nibbles), exact: the nibble with its
// sign bit flipped goes into the low mantissa of f16 1024 (1032 + q), then 1032 is subtracted
__device__ __forceinline__ uint32_t codes_pair_f16(uint32_t w, int i) {
  const uint32_t v = w >> (4 * i);
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(v), "n"(0x000F000F), "n"(0x64086408));
  __half2 r = *reinterpret_cast<__half2*>(&d);
  r = __hsub2(r, __floats2half2_rn(1032.0f, 1032.0f));
  return *reinterpret_cast<uint32_t*>(&r);
}

// q * s for a pair of exact codes and the fp16 scale: one f16 rounding
__device__ __forceinline__ uint32_t scale_pair(uint32_t q, __half2 s) {
  const __half2 r = __hmul2(*reinterpret_cast<__half2*>(&q), s);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Four int8 codes (bytes of w) times the scale, exactly, in fp32: the byte with its sign bit
// flipped (q + 128) becomes the low mantissa bits of 2^23 (fp32 2^23 + q + 128), the offset is
// subtracted exactly, and q * s has at most 8 + 11 significant bits.
__device__ __forceinline__ void codes8_scaled(uint32_t w, float s, float* v) {
  const uint32_t u = w ^ 0x80808080u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float f = __uint_as_float(prmt(u, 0x4B000000u, 0x7540u + i)) - 8388736.0f;
    v[i] = f * s;
  }
}

// Position of natural index i (0..7) inside a chunk stored in (0,4,1,5,2,6,3,7) order.
__device__ __forceinline__ int pair_pos(int i) { return i < 4 ? 2 * i : 2 * (i - 4) + 1; }

template <bool kGateUp, int kN, int kBits>
__global__ void __launch_bounds__((TcCfg<kGateUp, kN, kBits>::THREADS), 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_b,
                           const __grid_constant__ CUtensorMap tmap_c0,
                           const __grid_constant__ CUtensorMap tmap_c1, TcArgs a) {
  using C = TcCfg<kGateUp, kN, kBits>;
  static_assert(kBits == 4 || C::RING, "8-bit codes come through the code ring");
  constexpr int ST = C::STAGES;
  constexpr int RS = C::RING_STAGES > 0 ? C::RING_STAGES : 1;  // (1: unused without the ring)
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem + ST * C::STAGE_BYTES;  // [RS][matrix][128 rows][128 bytes] of codes
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + C::RING_STAGES * C::CODE_BYTES);
  uint64_t* full_a = bars;
  uint64_t* full_b = bars + ST;
  uint64_t* empty = bars + 2 * ST;
  uint64_t* acc_full = bars + 3 * ST;       // [2]
  uint64_t* acc_empty = bars + 3 * ST + 2;  // [2]
  uint64_t* drain = bars + 3 * ST + 4;      // abort path: completion of the issued MMAs
  uint64_t* cfull = bars + 3 * ST + 5;      // [RS] code slot landed
  uint64_t* cempty = cfull + RS;            // [RS] code slot read by the dequant warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cempty + RS);
  __shared__ int abort_flag_s;
  volatile int* abort_flag = &abort_flag_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      tc::mbar_init(full_a + s, C::DQW);
      tc::mbar_init(full_b + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full + b, 1);
      tc::mbar_init(acc_empty + b, 4);  // the 4 epilogue warps
    }
    tc::mbar_init(drain, 1);
    for (int s = 0; s < C::RING_STAGES; ++s) {
      tc::mbar_init(cfull + s, 1);
      tc::mbar_init(cempty + s, C::DQW);
    }
    tc::fence_barrier_init();
    abort_flag_s = 0;
  }
  if (warp == 2) {
    tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) tc::prefetch_tmap(&tmap_b);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_items = kGateUp ? a.hdr->n_items_gu : a.hdr->n_items_dn;
  const int nseg = a.hdr->nseg;
  const int nk = a.K / kTcBK;
  const int mtiles = a.Nw / kTcBM;
  auto A_of = [&](int s, int m) { return smem + s * C::STAGE_BYTES + m * C::A_BYTES; };
  auto B_of = [&](int s) { return smem + s * C::STAGE_BYTES + C::NMAT * C::A_BYTES; };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        TcTile t;
        tc_decode<kN>(a, item, nseg, mtiles, t);
        const int nbox = (t.nmma + C::BOX_ROWS - 1) / C::BOX_ROWS;  // only the rows the MMA reads
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % ST;
          const uint32_t ph = (it / ST) & 1;
          if (!tc::mbar_wait(empty + s, ph ^ 1, abort_flag, a.status)) { ok = false; break; }
          tc::mbar_arrive_expect_tx(full_b + s, nbox * C::BOX_BYTES);
          for (int bx = 0; bx < nbox; ++bx)
            tc::tma_load_2d(B_of(s) + bx * C::BOX_BYTES, &tmap_b, kb * kTcBK,
                            t.row0 + bx * C::BOX_ROWS, full_b + s);
        }
      }
      if (!ok)  // drain the copies that may still be in flight
        for (int j = (it > ST ? it - ST : 0); j < it; ++j)
          tc::mbar_wait_drain(full_b + (j % ST), (j / ST) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0, tcount = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++tcount) {
        TcTile t;
        tc_decode<kN>(a, item, nseg, mtiles, t);
        const uint32_t idesc = tc::idesc_f16(kTcBM, t.nmma);
        const int buf = tcount % C::NBUF;
        const uint32_t dtm = tmem + buf * C::ACC_COLS;
        // the epilogue has drained this buffer (the tile NBUF back)
        if (tcount >= C::NBUF && !tc::mbar_wait(acc_empty + buf, ((tcount / C::NBUF) - 1) & 1,
                                                abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % ST;
          const uint32_t ph = (it / ST) & 1;
          if (!tc::mbar_wait(full_a + s, ph, abort_flag, a.status) ||
              !tc::mbar_wait(full_b + s, ph, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint64_t da0 = tc::sw128_desc(tc::smem_u32(A_of(s, 0)));
          const uint64_t da1 = kGateUp ? tc::sw128_desc(tc::smem_u32(A_of(s, 1))) : 0;
          const uint64_t db = tc::sw128_desc(tc::smem_u32(B_of(s)));
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk) {
            const uint32_t acc = (kb | kk) ? 1u : 0u;
            // +32 bytes per 16-wide K step inside the swizzle row (address field is in 16 B)
            tc::mma_f16_ss(dtm, da0 + 2 * kk, db + 2 * kk, idesc, acc);
            if (kGateUp) tc::mma_f16_ss(dtm + kN, da1 + 2 * kk, db + 2 * kk, idesc, acc);
          }
          tc::mma_commit(empty + s);
        }
        if (!ok) break;
        tc::mma_commit(acc_full + buf);
      }
      if (!ok) {  // drain every MMA issued so far before TMEM is released
        tc::mma_commit(drain);
        tc::mbar_wait_drain(drain, 0);
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------------ code ring producer
    if (C::RING && lane == 0) {
      tc::prefetch_tmap(&tmap_c0);
      if (kGateUp) tc::prefetch_tmap(&tmap_c1);
      int cit = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        TcTile t;
        tc_decode<kN>(a, item, nseg, mtiles, t);
        const int32_t wrow = t.e * a.Nw + t.mt * kTcBM;
        for (int kb = 0; kb < nk; kb += C::SLOT_K, ++cit) {
          const int cs = cit % RS;
          if (!tc::mbar_wait(cempty + cs, ((cit / RS) & 1) ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          // the dequant warps read the slot through the generic proxy, the TMA below rewrites it
          // through the async proxy: a cross-proxy fence orders the two
          tc::fence_proxy_async_smem();
          // a slot past the end of the row (nk not a multiple of SLOT_K) reads zero fill
          uint8_t* dst = ring + cs * C::CODE_BYTES;
          tc::mbar_arrive_expect_tx(cfull + cs, C::CODE_BYTES);
          tc::tma_load_2d(dst, &tmap_c0, kb * C::STAGE_CODE_BYTES, wrow, cfull + cs);
          if (kGateUp)
            tc::tma_load_2d(dst + C::CODE_BYTES / 2, &tmap_c1, kb * C::STAGE_CODE_BYTES, wrow,
                            cfull + cs);
        }
      }
      if (!ok)  // drain the copies that may still be in flight
        for (int j = (cit > RS ? cit - RS : 0); j < cit; ++j)
          tc::mbar_wait_drain(cfull + (j % RS), (j / RS) & 1);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + C::DQW) {
    // ------------------------------------------------------------------ dequant producers
    // SUBS threads per weight row and matrix, each converting CPT of the stage's eight 8-code
    // chunks: 16 warps on 256-row gate/up tiles (2 x 4 chunks), 8 warps elsewhere (gate/up
    // 1 x 8, down 2 x 4)
    constexpr int SUBS = (C::DQW * 32) / (C::NMAT * kTcBM);  // threads per row
    constexpr int CPT = 8 / SUBS;                              // chunks per thread and stage
    constexpr int TB = kBits * CPT;       // bytes of codes per thread and stage: 8 .. 64
    constexpr int NV = TB >= 16 ? TB / 16 : 1;  // 16-byte vectors of them (8 bytes: one half)
    const int pt = threadIdx.x - 128;
    const int sub = pt % SUBS;
    const int rr = pt / SUBS;             // gate/up: matrix x 128 + row; down: row
    const int mat = kGateUp ? (rr >> 7) : 0;
    const int r = rr & 127;
    const uint8_t* codes = mat ? a.codes1 : a.codes0;
    const __half* scales = mat ? a.scales1 : a.scales0;
    const int64_t row_bytes = static_cast<int64_t>(a.K) * kBits / 8;
    const int64_t srow = a.K / a.group;
    // scale of stage kb (64 codes): group (64 kb) / G
    const int gs = a.group == 64 ? 0 : a.group == 128 ? 1 : 2;
    // ring: this thread's weight row inside a slot (128 bytes: SLOT_K stages, 16-byte chunks
    // swizzled as c ^ (r % 8))
    const int roff = (kGateUp ? mat * (C::CODE_BYTES / 2) : 0) + r * 128;
    int it = 0, cit = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      TcTile t;
      tc_decode<kN>(a, item, nseg, mtiles, t);
      const int64_t wrow = static_cast<int64_t>(t.e) * a.Nw + t.mt * kTcBM + r;
      const uint8_t* cp = codes + wrow * row_bytes + sub * TB;
      const __half* sp = scales + wrow * srow;
      const uint32_t soff = (r >> 3) * 1024 + (r & 7) * 128;
      // codes (and scales) of the next 4 stages stay in flight in fixed register slots: the loop
      // is unrolled by 4 so slot u is refilled for stage kb + 4 right after stage kb used it
      // (the 256-row kernel; the 64-row kernel reads its codes from the TMA ring)
      constexpr int PD = 4;
      constexpr int NVG = C::RING ? 1 : NV;  // register vectors of the global-load path
      uint4 cA[PD][NVG];
      // scale of stage kb's group, kept as raw fp16 bits: converting on load would make the load
      // complete right away
      unsigned short sc[PD];
      auto ld = [&](int kb, uint4 (&x)[NVG]) {
        if (!C::RING && kb < nk) {
          const uint8_t* src = cp + static_cast<int64_t>(kb) * (kTcBK * kBits / 8);
          if (TB >= 16) {
#pragma unroll
            for (int v = 0; v < NVG; ++v) x[v] = __ldg(reinterpret_cast<const uint4*>(src) + v);
          } else {
            const uint2 h = __ldg(reinterpret_cast<const uint2*>(src));
            x[0] = make_uint4(h.x, h.y, 0u, 0u);
          }
        }
      };
#pragma unroll
      for (int u = 0; u < PD; ++u) {
        ld(u, cA[u]);
        if (u < nk) sc[u] = __ldg(reinterpret_cast<const unsigned short*>(sp) + (u >> gs));
      }
      for (int kb0 = 0; ok && kb0 < nk; kb0 += PD) {
#pragma unroll
        for (int u = 0; u < PD; ++u) {
          const int kb = kb0 + u;
          if (kb >= nk) break;
          const int s = it % ST;
          const uint32_t ph = (it / ST) & 1;
          // scale of this stage's group (fp16), and as fp32 for the exact 8-bit products
          const __half sh = __ushort_as_half(sc[u]);
          const __half2 s2 = __halves2half2(sh, sh);
          const float sf = __half2float(sh);
          uint4 xv[NV];
          if (C::RING) {
            const int cs = cit % RS;
            const int ks = kb % C::SLOT_K;
            if (ks == 0 && !tc::mbar_wait(cfull + cs, (cit / RS) & 1, abort_flag, a.status)) {
              ok = false;
              break;
            }
            const uint8_t* src = ring + cs * C::CODE_BYTES + roff;
            // byte offset of this thread's piece inside the slot row (unswizzled), then the
            // 16-byte chunk it starts in and the offset inside that chunk
            const int boff = ks * (kTcBK * kBits / 8) + sub * TB;
            const int ch = boff >> 4, inb = boff & 15;
            if (TB >= 16) {
#pragma unroll
              for (int v = 0; v < NV; ++v)
                xv[v] = *reinterpret_cast<const uint4*>(src + (((ch + v) ^ (r & 7)) << 4));
            } else {
              const uint2 h = *reinterpret_cast<const uint2*>(src + ((ch ^ (r & 7)) << 4) + inb);
              xv[0] = make_uint4(h.x, h.y, 0u, 0u);
            }
            if (ks == C::SLOT_K - 1 || kb == nk - 1) {
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(cempty + cs);  // the slot's codes are all read
              ++cit;
            }
          } else {
#pragma unroll
            for (int v = 0; v < NV; ++v) xv[v] = cA[u][v < NVG ? v : 0];
            ld(kb + PD, cA[u]);
          }
          if (kb + PD < nk)
            sc[u] = __ldg(reinterpret_cast<const unsigned short*>(sp) + ((kb + PD) >> gs));
          if (!tc::mbar_wait(empty + s, ph ^ 1, abort_flag, a.status)) { ok = false; break; }
          uint8_t* dst = A_of(s, mat) + soff;
          // the codes as words: 4-bit one word per 8-code chunk, 8-bit two
          uint32_t wd[4 * NV];
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            wd[4 * v] = xv[v].x; wd[4 * v + 1] = xv[v].y; wd[4 * v + 2] = xv[v].z; wd[4 * v + 3] = xv[v].w;
          }
          if (kBits == 8) {
            // 8 codes (bytes m0..m7, natural order) per chunk -> f16 pairs (m0,m4) (m1,m5)
            // (m2,m6) (m3,m7); q * s is exact in fp32 and rounded once to f16
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
              float v[8];
              codes8_scaled(wd[2 * j], sf, v);
              codes8_scaled(wd[2 * j + 1], sf, v + 4);
              uint4 o;
              o.x = f32x2_to_f16x2_sat(v[0], v[4]);
              o.y = f32x2_to_f16x2_sat(v[1], v[5]);
              o.z = f32x2_to_f16x2_sat(v[2], v[6]);
              o.w = f32x2_to_f16x2_sat(v[3], v[7]);
              const int chunk = sub * CPT + j;
              *reinterpret_cast<uint4*>(dst + ((chunk ^ (r & 7)) << 4)) = o;
            }
          } else {
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
              const uint32_t w = wd[j];
              uint4 o;
              o.x = scale_pair(codes_pair_f16(w, 0), s2);
              o.y = scale_pair(codes_pair_f16(w, 1), s2);
              o.z = scale_pair(codes_pair_f16(w, 2), s2);
              o.w = scale_pair(codes_pair_f16(w, 3), s2);
              const int chunk = sub * CPT + j;
              *reinterpret_cast<uint4*>(dst + ((chunk ^ (r & 7)) << 4)) = o;
            }
          }
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(full_a + s);
          ++it;
        }
      }
      if (!ok) break;
    }
    __syncwarp();
  } else if (warp >= 4 + C::DQW) {
    // ------------------------------------------------------------------ epilogue
    const int q4 = warp & 3;  // TMEM lane quarter of this warp
    int tcount = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++tcount) {
      TcTile t;
      tc_decode<kN>(a, item, nseg, mtiles, t);
      const int buf = tcount % C::NBUF;
      if (!tc::mbar_wait(acc_full + buf, (tcount / C::NBUF) & 1, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      const int irow = t.mt * kTcBM + q4 * 32 + lane;  // weight row = output column
      const uint32_t lane_addr = tmem + buf * C::ACC_COLS + (static_cast<uint32_t>(q4 * 32) << 16);
      // 16 token columns at a time (the registers of 768-thread CTAs are few)
      for (int c = 0; c < t.nmma; c += 16) {
        uint32_t g[16];
        tc::tmem_ld16(lane_addr + c, g);
        // range exponents of this chunk's token rows (the B rows were stored times 2^-e)
        const int n_here = min(16, t.nvalid - c);
        const int my_e = (a.aexp && lane < n_here) ? a.aexp[t.row0 + c + lane] : 0;
        if (kGateUp) {
          uint32_t u[16];
          tc::tmem_ld16(lane_addr + kN + c, u);
          tc::tmem_ld_wait();
          __half* h = static_cast<__half*>(a.out);
          const int col = (irow & ~7) | pair_pos(irow & 7);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = c + j;
            const int e = __shfl_sync(0xffffffffu, my_e, j);
            if (n < t.nvalid) {
              // h stored times 2^-2e (gate and up are at scale 2^-e each)
              const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
              h[static_cast<int64_t>(t.row0 + n) * a.Nw + col] =
                  f32_to_f16_sat(silu_scaled(gv, exp2i(e)) * uv);
            }
          }
          if (a.hexp && t.mt == 0 && q4 == 0 && lane < n_here) a.hexp[t.row0 + c + lane] = 2 * my_e;
        } else {
          tc::tmem_ld_wait();
          float* y = static_cast<float*>(a.out);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = c + j;
            const float up = exp2i(__shfl_sync(0xffffffffu, my_e, j));
            if (n < t.nvalid)
              y[static_cast<int64_t>(t.row0 + n) * a.Nw + irow] = __uint_as_float(g[j]) * up;
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty + buf);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ----------------------------------------------------------------------------- gather

// xp[r] = x[perm[r]], each 8-wide chunk reordered for the GEMM that reads it (kMode):
//   0: bf16 in (0,4,1,5,2,6,3,7) order (the per-warp decode GEMM)
//   1: f16 with element i at position bitrev3(i) (the CTA-staged decode GEMM)
//   2: f16 in (0,4,1,5,2,6,3,7) order (the tensor-core GEMM)
// f16 is exact from bf16 within its range and saturated at +-65504 outside it.
template <int kMode>
__global__ void __launch_bounds__(128) gather_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const int* __restrict__ perm, int H,
                                                          uint16_t* __restrict__ xp,
                                                          int* __restrict__ rexp) {
  const int row = blockIdx.x;
  const int tok = perm[row];
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(tok) * H);
  uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<int64_t>(row) * H);
  float s = 1.0f;
  if (kMode != 0) {
    // the row's range exponent (f16 copies): its largest magnitude, then 2^-e
    __shared__ uint32_t wmag[4];
    uint32_t m = 0;
    for (int c = threadIdx.x; c < H / 8; c += blockDim.x) m = max(m, bf16x8_mag(__ldg(src + c)));
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) wmag[threadIdx.x >> 5] = m;
    __syncthreads();
    const int e = range_exp(max(max(wmag[0], wmag[1]), max(wmag[2], wmag[3])));
    if (threadIdx.x == 0 && rexp) rexp[row] = e;
    s = exp2i(-e);
  }
  for (int c = threadIdx.x; c < H / 8; c += blockDim.x) {
    const uint4 v = __ldg(src + c);
    uint4 o;
    if (kMode == 1) {
      o = bf16_chunk_to_f16_pairs(v, s);
    } else if (kMode == 2) {
      o.x = f32x2_to_f16x2_sat(bf16_lo_f32(v.x) * s, bf16_lo_f32(v.z) * s);  // x0, x4
      o.y = f32x2_to_f16x2_sat(bf16_hi_f32(v.x) * s, bf16_hi_f32(v.z) * s);  // x1, x5
      o.z = f32x2_to_f16x2_sat(bf16_lo_f32(v.y) * s, bf16_lo_f32(v.w) * s);  // x2, x6
      o.w = f32x2_to_f16x2_sat(bf16_hi_f32(v.y) * s, bf16_hi_f32(v.w) * s);  // x3, x7
    } else {
      o.x = prmt(v.x, v.z, 0x5410);  // x0, x4
      o.y = prmt(v.x, v.z, 0x7632);  // x1, x5
      o.z = prmt(v.y, v.w, 0x5410);  // x2, x6
      o.w = prmt(v.y, v.w, 0x7632);  // x3, x7
    }
    dst[c] = o;
  }
}

cudaError_t launch_gather_rows(const void* x, const int* perm, int64_t rows, int64_t H, void* xp,
                               int mode, int* rexp, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const unsigned g = static_cast<unsigned>(rows);
  const __nv_bfloat16* xs = static_cast<const __nv_bfloat16*>(x);
  uint16_t* xd = static_cast<uint16_t*>(xp);
  const int h = static_cast<int>(H);
  if (mode == 1)
    gather_rows_kernel<1><<<g, 128, 0, stream>>>(xs, perm, h, xd, rexp);
  else if (mode == 2)
    gather_rows_kernel<2><<<g, 128, 0, stream>>>(xs, perm, h, xd, rexp);
  else
    gather_rows_kernel<0><<<g, 128, 0, stream>>>(xs, perm, h, xd, nullptr);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- host

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Row-major f16 [rows, cols]: boxes of box_rows rows x 64 columns, 128-byte swizzle, zero fill.
static bool make_row_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
                          int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {kTcBK, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Codes [rows, row_bytes] (K/2 for 4-bit codes, K for 8-bit): boxes of 128 bytes x 128 weight
// rows, 128-byte swizzle, zero fill past the row end.
static bool make_code_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {128, kTcBM};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kGateUp, int kN, int kBits>
cudaError_t launch_gemm_tc_t(const TcArgs& a, const void* b_rows, int64_t rows, int64_t experts,
                             int num_sms, cudaStream_t stream) {
  using C = TcCfg<kGateUp, kN, kBits>;
  CUtensorMap map, c0, c1;
  if (!make_row_tmap(&map, b_rows, rows, a.K, C::BOX_ROWS)) return cudaErrorInvalidValue;
  c0 = map;
  c1 = map;
  if (C::RING) {
    const int64_t row_bytes = static_cast<int64_t>(a.K) * kBits / 8;
    if (!make_code_tmap(&c0, a.codes0, experts * a.Nw, row_bytes)) return cudaErrorInvalidValue;
    if (kGateUp && !make_code_tmap(&c1, a.codes1, experts * a.Nw, row_bytes))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_tc_kernel<kGateUp, kN, kBits>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  grouped_gemm_tc_kernel<kGateUp, kN, kBits><<<num_sms, C::THREADS, C::SMEM, stream>>>(map, c0, c1,
                                                                                         a);
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const TcArgs& a, bool gate_up, const void* b_rows, int64_t rows,
                           int64_t experts, int tile_rows, int num_sms, cudaStream_t stream) {
  if (a.bits == 8) {  // 8-bit codes: 64-row tiles (the code ring) only
    if (tile_rows != kTcRowsSmall) return cudaErrorInvalidValue;
    return gate_up ? launch_gemm_tc_t<true, kTcRowsSmall, 8>(a, b_rows, rows, experts, num_sms, stream)
                   : launch_gemm_tc_t<false, kTcRowsSmall, 8>(a, b_rows, rows, experts, num_sms, stream);
  }
  if (tile_rows == kTcRowsSmall)
    return gate_up ? launch_gemm_tc_t<true, kTcRowsSmall, 4>(a, b_rows, rows, experts, num_sms, stream)
                   : launch_gemm_tc_t<false, kTcRowsSmall, 4>(a, b_rows, rows, experts, num_sms, stream);
  if (tile_rows != kTcRows) return cudaErrorInvalidValue;
  return gate_up ? launch_gemm_tc_t<true, kTcRows, 4>(a, b_rows, rows, experts, num_sms, stream)
                 : launch_gemm_tc_t<false, kTcRows, 4>(a, b_rows, rows, experts, num_sms, stream);
}

}  // namespace strata
