// K4 (decode path): W4A16 grouped GEMM for segments with few rows, where the layer is bound by
// streaming the activated experts' int4 weights from HBM. One launch covers every expert's group
// ("Strata" 3090 tuning, xdnf.cn/news/329730, §3.2: one grouped GEMM instead of one GEMM launch per
// expert); dequantization happens in registers ("Strata" architecture essay, dpshk.com/news/6309482,
// §3.2: decode is bandwidth-bound, so use wide loads and keep the small operands close).
//
// Work item = (8-row chunk of one expert's rows, block of weight rows, contraction split). A
// persistent CTA (two per SM) has one producer warp and 8 consumer warps sharing a ring of stages;
// a stage holds one 128-wide contraction group of the block:
//  * weights: gate/up 128 gate + 128 up rows, down 256 rows, 64 bytes each, by one TMA box per
//    matrix (canonical row-major codes, no re-layout);
//  * activations: the chunk's 8 rows x 128 bf16, gathered through the routing permutation by
//    cp.async, 16-byte pieces swizzled so that the consumers' fragment loads do not conflict;
//  * scales: when the scale rows allow it (row stride and base 16-byte aligned), one TMA box per
//    matrix of 16 bytes (8 consecutive groups, the aligned run holding the stage's group) x rows;
//    otherwise the fp16 pair holding each row's scale, by 4-byte cp.async. Either way they land
//    on the stage's own full barrier.
// The producer streams stages ahead (mbarrier full/empty pairs; every wait is time-bounded) while
// the consumers compute; consumer warp w owns 16 gate + 16 up rows (gate/up) or 32 rows (down).
//
// A consumer warp computes with mma.sync m16n8k16 (bf16 in, fp32 accumulate) and swapped operands:
// weight rows are the A operand, the (up to 8) tokens the B operand.
//  * Lane (g = lane/4, t = lane%4) takes 16 bytes = 32 codes of rows g and g+8 per group, and the
//    contraction order inside the group is permuted so that they feed exactly the lane's A-fragment
//    slots. The activations are stored with element i of every 8-wide chunk at position bitrev3(i),
//    i.e. as words (x0,x4) (x2,x6) (x1,x5) (x3,x7) (x by the router or the row gather, h by the
//    gate/up epilogue): one 16-byte load gives the B-fragment pairs of both nibble planes of an MMA
//    step in adjacent registers. A dot product does not depend on the order of its terms, so no
//    weight re-layout is needed.
//  * The MMAs take f16 operands: the activations the decode path stages are f16, converted exactly
//    from bf16 (saturated at +-65504). int4 -> f16 takes one LOP3 per code pair and one shift per
//    8 codes: each word's nibbles 0/4 and 2/6 (after >> 8) become f16 1032 + q (the nibble in the
//    low mantissa bits of 1024), nibbles 1/5 and 3/7 become 72 + q without a shift (the nibble in
//    mantissa bits 4-7 of 64, where they weigh 1). The low planes multiply the activation pairs
//    (x0,x4), (x2,x6), the high planes (x1,x5), (x3,x7), both into one accumulator per tile; one
//    correction accumulator (MMAs with A = 1032 and A = 72, shared by both tiles) removes the
//    offsets, and the group's fp16 scale is applied in fp32: acc += s * (P - C). Each group's
//    first MMAs start from zero, so nothing is cleared per group. Weights are never rounded.
//  * Small batches split the contraction; the last split to arrive (device counter per warp tile)
//    sums the partials in split order and applies the epilogue, so results stay deterministic.
//  * The smallest batches (at most two tiles per CTA, tile = chunk x row block) take the kEven
//    schedule instead: the launch's stages (tiles x K/128, tiles in chunk-fastest order) are cut
//    into one equal contiguous range per CTA, so that every CTA streams the same weight bytes. A
//    tile whose stages fall into two or more CTAs' ranges is split; its pieces publish partial
//    sums in per-CTA slots (a CTA has at most two split pieces: its range's first and last) and
//    the last piece to arrive sums them in piece order. With more tiles per CTA, claiming
//    whole tiles is faster: a CTA that streams faster takes more.
// Gate/up writes h = silu(u) * v (bf16); down writes y (fp32) for the combine.
#include <cudaTypedefs.h>

#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace strata {
namespace {

constexpr int kCW = 8;                     // consumer warps
constexpr int kThreads = (kCW + 1) * 32;   // + one producer warp
constexpr int kStages = 5;
constexpr int kWBytes = 16384;             // weights of one stage (256 rows x 64 bytes)
constexpr int kActOff = kWBytes;           // 8 rows x 256 bytes
constexpr int kScOff = kActOff + 2048;     // 256 rows x 4 bytes (cp.async) or 16 bytes (TMA)
constexpr int kCtasPerSm = 2;
// Stage layout with scales copied as 4-byte pairs (kScTma false) or as 16-byte TMA rows (true).
template <bool kScTma>
struct CtaLayout {
  static constexpr int kScRowBytes = kScTma ? 16 : 4;
  static constexpr int kHdrOff = kScOff + 256 * kScRowBytes;
  static constexpr int kStageBytes = kScTma ? 22656 : 19584;  // 128-byte multiple >= header end
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kSmemBytes = kBarOff + 2 * kStages * 8 + 16;
};
constexpr int kBlockK = 128;               // contraction per stage

struct StageHdr {
  int e, rbase, nvalid, blk, ks, cidx;  // item: expert, first GEMM row, rows, row block, split, chunk
  int g, gbeg, gend;                    // this stage's group and the item's group range
  int done;                             // no more items
  int split;                            // kEven: the piece's split word (split_np, split_slot)
};
static_assert(CtaLayout<false>::kHdrOff + static_cast<int>(sizeof(StageHdr)) <=
                  CtaLayout<false>::kStageBytes,
              "stage layout");
static_assert(CtaLayout<true>::kHdrOff + static_cast<int>(sizeof(StageHdr)) <=
                  CtaLayout<true>::kStageBytes,
              "stage layout");
static_assert(kCtasPerSm * (CtaLayout<true>::kSmemBytes + 1024) <= 228 * 1024,
              "two CTAs per SM");

// int4 -> f16 in one LOP3 per code pair, d = (v & mask) ^ c: the masked nibbles land in the
// mantissa with their sign bit flipped. Nibbles at bits 0-3 / 16-19 go into the low mantissa bits
// of f16 1024 and give 1032 + q; nibbles at bits 4-7 / 20-23 go into mantissa bits 4-7 of f16 64,
// where one step is worth 1, and give 72 + q. Both are exact.
__device__ __forceinline__ uint32_t nib_lo_f16(uint32_t v) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(v), "n"(0x000F000F), "n"(0x64086408));
  return d;
}
__device__ __forceinline__ uint32_t nib_hi_f16(uint32_t v) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(v), "n"(0x00F000F0), "n"(0x54805480));
  return d;
}

__device__ __forceinline__ void cp_async4(uint32_t saddr, const void* gmem, bool pred, uint64_t pol) {
  const int sz = pred ? 4 : 0;
  asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 4, %2, %3;\n" ::"r"(saddr),
               "l"(gmem), "r"(sz), "l"(pol));
}
__device__ __forceinline__ void cp_async16s(uint32_t saddr, const void* gmem, bool pred) {
  const int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(saddr), "l"(gmem), "r"(sz));
}
// The barrier receives one arrival once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar))
               : "memory");
}

// Group sizes: the weights of a stage are one 128-wide contraction block. With 128-wide or 256-wide
// scale groups (kG) the block has one scale per row; with 64-wide groups it has two, and lane t then
// takes codes 16t..16t+15 of each 64-half (instead of 32t..32t+31 of the block) so that MMAs j = 0,1
// stay inside the first group and j = 2,3 inside the second.
//
// Activation piece (16 bytes = 8 values) that feeds MMA step j of lane t.
template <int kG>
__device__ __forceinline__ int act_piece(int t, int j) {
  return kG == 64 ? (j < 2 ? 2 * t + j : 8 + 2 * t + (j - 2)) : 4 * t + j;
}
// Position of 16-byte piece q (0..15) of activation row n inside the row. A 128-bit shared load
// is served 8 lanes at a time: lanes 8p..8p+7 read rows 2p, 2p+1, pieces act_piece(t, c) for
// t = 0..3 and a fixed c. The map sends those 8 pieces to 8 different 16-byte bank groups, so
// the loads do not conflict.
template <int kG>
__device__ __forceinline__ int act_swz(int n, int q) {
  return kG == 64 ? q ^ (n & 1) : q ^ ((q >> 3) & 1) ^ ((n & 1) << 1);
}

// kEven schedule. The CTA whose stage range holds stage u, the ranges being [c W / C, (c + 1) W / C)
// for c = 0 .. C - 1 with C <= W (no range is empty): the largest c with c W / C <= u.
__device__ __forceinline__ int cta_of_stage(int u, int W, int C) {
  return static_cast<int>(((static_cast<int64_t>(u) + 1) * C + W - 1) / W) - 1;
}
// A piece's split word: bits 0-11 the tile's first CTA c0, bits 12-23 the tile's pieces np (CTAs
// c0 .. c0 + np - 1; 1 = not split), bit 24 set when the piece is not its CTA's first (its slot is
// then 2 cta + 1, else 2 cta), bit 25 set when the tile's first piece is not c0's first piece (its
// slot is then 2 c0 + 1, else 2 c0); the later pieces are their CTAs' first (slots 2 c). A launch
// has at most 4096 CTAs (checked on the host), so c0 and np fit.
__device__ __forceinline__ int split_np(int w) { return (w >> 12) & 0xFFF; }
__device__ __forceinline__ int split_slot(int w, int pc) {
  const int c = (w & 0xFFF) + pc;
  return 2 * c + (pc == 0 ? (w >> 25) & 1 : 0);
}

struct CtaGemmParams {
  GemmArgs a;
  int nblk;   // row blocks per expert
  int RB;     // rows per block (gate/up: per matrix)
};

// map0/map1: codes of gate (or down) / up; smap0/smap1: their scales (kScTma only).
// kEven: the equal-stage-range schedule of the smallest batches (see above).
template <bool kGateUp, int kG, bool kScTma, bool kEven>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    grouped_gemm_cta_kernel(const __grid_constant__ CUtensorMap map0,
                            const __grid_constant__ CUtensorMap map1,
                            const __grid_constant__ CUtensorMap smap0,
                            const __grid_constant__ CUtensorMap smap1, const CtaGemmParams p) {
  using Lay = CtaLayout<kScTma>;
  constexpr int kHdrOff = Lay::kHdrOff;
  constexpr int kStageBytes = Lay::kStageBytes;
  constexpr int kBarOff = Lay::kBarOff;
  extern __shared__ __align__(1024) unsigned char smem[];
  const GemmArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);
  uint32_t* status = &a.hdr->status;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1 + 32);  // producer expect_tx arrival + 32 cp.async arrivals
      tc::mbar_init(&empty[s], kCW);    // one arrival per consumer warp
    }
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();

  const int ngroups = a.K / kBlockK;
  const int KS = a.ksplit;

  if (warp == kCW) {
    // ------------------------------------------------------------------ producer warp
    if (lane == 0) {
      tc::prefetch_tmap(&map0);
      if (kGateUp) tc::prefetch_tmap(&map1);
      if (kScTma) {
        tc::prefetch_tmap(&smap0);
        if (kGateUp) tc::prefetch_tmap(&smap1);
      }
    }
    if (kGateUp) griddep_wait();  // the work lists and x come from the router
    griddep_launch();
    int* const next_ctr = kGateUp ? &a.hdr->next_gu : &a.hdr->next_dn;
    const int n_items = kGateUp ? a.hdr->n_items_gu : a.hdr->n_items_dn;
    const int nchunks = a.hdr->n_chunks;
    const int64_t srow = a.K / kG;                // scale row stride (fp16)
    const int q = lane & 15;                      // activation piece of this lane
    // weights (64 bytes per row) and, with kScTma, scales (16 bytes per row) of the stage
    constexpr uint32_t kRowTx = 64u + (kScTma ? 16u : 0u);
    const uint32_t tx_bytes = kGateUp ? 2u * p.RB * kRowTx : static_cast<uint32_t>(p.RB) * kRowTx;
    int stage = 0;
    uint32_t phase = 0;
    bool waited = kGateUp;  // down: griddep_wait still pending (h comes from gate/up)
    int npend = 0;          // down, first item: stages whose activation copies wait for it
    bool ok = true;
    if constexpr (!kEven) {
    int item = 0;
    if (lane == 0) item = atomicAdd(next_ctr, 1);
    item = __shfl_sync(0xffffffffu, item, 0);
    while (item < n_items && ok) {
      int nxt = 0;
      if (lane == 0) nxt = atomicAdd(next_ctr, 1);
      const int cidx = item % nchunks;
      const int rest = item / nchunks;
      const int blk = rest % p.nblk;
      const int ks = rest / p.nblk;
      const int4 ch = __ldg(a.chunk_list + cidx);
      const int e = ch.x, rbase = ch.y, nvalid = ch.z;
      const int gbeg = (ks * ngroups) / KS, gend = ((ks + 1) * ngroups) / KS;
      const int64_t wrow0 = static_cast<int64_t>(e) * a.N + static_cast<int64_t>(blk) * p.RB;
      // activation rows of this lane's pieces: n = 2 i + lane / 16
      const __nv_bfloat16* arow[4];
      bool avalid[4];
      // down: h rows come from gate/up (wait for it before the first activation copy)
      for (int g = gbeg; g < gend; ++g) {
        if (!tc::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
        // The consumers read the slot through the generic proxy; the TMA boxes below write it
        // through the async proxy. The empty barrier orders those reads before this point, and
        // this cross-proxy fence orders them before the new boxes (without it, a warp's loads of
        // the slot's first rows could return the next stage's bytes, about one forward in 100).
        tc::fence_proxy_async_smem();
        unsigned char* st = smem + stage * kStageBytes;
        // weights and scales are read once per call: evict them from L2 first (made here, per
        // stage, so that the policy holds no register across the loop)
        const uint64_t pol = l2_evict_first_policy();
        if (lane == 0) {
          StageHdr* h = reinterpret_cast<StageHdr*>(st + kHdrOff);
          h->e = e; h->rbase = rbase; h->nvalid = nvalid; h->blk = blk; h->ks = ks; h->cidx = cidx;
          h->g = g; h->gbeg = gbeg; h->gend = gend; h->done = 0;
          tc::mbar_arrive_expect_tx(&full[stage], tx_bytes);
          tc::tma_load_2d_hint(st, &map0, g * 64, static_cast<int32_t>(wrow0), &full[stage], pol);
          if (kGateUp)
            tc::tma_load_2d_hint(st + p.RB * 64, &map1, g * 64, static_cast<int32_t>(wrow0),
                                 &full[stage], pol);
          if (kScTma) {
            // the aligned run of 8 scale groups holding this stage's group(s): 16 bytes per row
            const int sx = (kG == 64 ? 2 * g : kG == 128 ? g : g >> 1) & ~7;
            tc::tma_load_2d_hint(st + kScOff, &smap0, sx, static_cast<int32_t>(wrow0),
                                 &full[stage], pol);
            if (kGateUp)
              tc::tma_load_2d_hint(st + kScOff + p.RB * 16, &smap1, sx,
                                   static_cast<int32_t>(wrow0), &full[stage], pol);
          }
        }
        // scales: the 4-byte fp16 pair holding group g, 8 rows per lane
        // 4-byte scale pair holding this block's scale(s): groups 2g, 2g+1 (kG = 64), g (128) or
        // g / 2 (256), the pair starting at an even group
        const int gp = kG == 64 ? 2 * g : kG == 128 ? (g & ~1) : ((g >> 1) & ~1);
#pragma unroll
        for (int i = 0; i < (kScTma ? 0 : 8); ++i) {
          const int r = lane + 32 * i;  // stage scale row
          const __half* sbase;
          int64_t row;
          if (kGateUp) {
            sbase = r < p.RB ? a.scales0 : a.scales1;
            row = wrow0 + (r < p.RB ? r : r - p.RB);
          } else {
            sbase = a.scales0;
            row = wrow0 + r;
          }
          const bool in = kGateUp ? true : (blk * p.RB + r < a.N);
          cp_async4(tc::smem_u32(st + kScOff + r * 4), sbase + (in ? row : wrow0) * srow + gp, in,
                    pol);
        }
        if (g == gbeg) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = 2 * i + (lane >> 4);
            avalid[i] = n < nvalid;
            int64_t src = rbase + (avalid[i] ? n : 0);
            if (a.perm) src = __ldg(a.perm + src);
            arow[i] = a.act + src * a.K;
          }
        }
        auto issue_act = [&](int gg, unsigned char* sst, uint64_t* bar) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = 2 * i + (lane >> 4);
            const uint32_t dst = tc::smem_u32(sst + kActOff + n * 256 + (act_swz<kG>(n, q) << 4));
            cp_async16s(dst, reinterpret_cast<const char*>(arow[i] + gg * kBlockK) + q * 16,
                        avalid[i]);
          }
          cp_async_arrive_noinc(bar);
        };
        if (waited) {
          issue_act(g, st, &full[stage]);
        } else {
          // down, first item: weights and scales of up to kStages groups go out before waiting
          // for gate/up (which writes h); their activation copies follow the wait
          ++npend;
          if (npend == kStages || g == gend - 1) {
            griddep_wait();
            waited = true;
            int s0 = stage - (npend - 1);
            if (s0 < 0) s0 += kStages;
            for (int j = 0; j < npend; ++j) {
              const int ss = (s0 + j) % kStages;
              issue_act(g - (npend - 1) + j, smem + ss * kStageBytes, &full[ss]);
            }
          }
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      item = __shfl_sync(0xffffffffu, nxt, 0);
    }
    } else {
    // (This branch repeats the stage loop above instead of sharing it: one loop serving both
    // schedules made the claimed-tile path slower at 16 tokens, gate/up +2 us of 88.6.)
    // this CTA's stage range; C = the CTAs that get a range (each at least one stage); the host
    // takes this schedule only for launches with at most two tiles per CTA, so W is small
    const int W = nchunks * p.nblk * ngroups;
    const int C = W < static_cast<int>(gridDim.x) ? W : static_cast<int>(gridDim.x);
    const int cta = blockIdx.x;
    constexpr int kRB = kGateUp ? kCW * 16 : kCW * 32;  // p.RB as a constant
    int u = cta < C ? static_cast<int>(static_cast<int64_t>(cta) * W / C) : 0;
    const int u_end = cta < C ? static_cast<int>(static_cast<int64_t>(cta + 1) * W / C) : 0;
    bool first_piece = true;
    while (u < u_end && ok) {
      // the piece: stages [gbeg, gend) of tile `tile`
      const int tile = u / ngroups;
      const int t0u = tile * ngroups;  // the tile's first stage
      const int gbeg = u - t0u;
      const int gend = u_end - t0u < ngroups ? u_end - t0u : ngroups;
      // CTAs c0 .. c0 + np - 1 hold the tile's pieces; each CTA's range is contiguous, so a CTA
      // has a split tile only as its first piece (slot 2 cta) and its last (slot 2 cta + 1)
      const int c0 = cta_of_stage(t0u, W, C);
      const int np = cta_of_stage(t0u + ngroups - 1, W, C) - c0 + 1;
      const int split = c0 | (np << 12) | (first_piece ? 0 : 1 << 24) |
                        (static_cast<int64_t>(c0) * W / C == t0u ? 0 : 1 << 25);
      first_piece = false;
      u = t0u + gend;
      const int cidx = tile % nchunks;
      const int blk = tile / nchunks;
      const int4 ch = __ldg(a.chunk_list + cidx);
      const int e = ch.x, rbase = ch.y, nvalid = ch.z;
      const int64_t wrow0 = static_cast<int64_t>(e) * a.N + static_cast<int64_t>(blk) * kRB;
      // activation rows of this lane's pieces (n = 2 i + lane / 16) and which of them are live
      int arow[4];
      unsigned amask = 0;
      // down: h rows come from gate/up (wait for it before the first activation copy)
      for (int g = gbeg; g < gend; ++g) {
        if (!tc::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, status)) { ok = false; break; }
        // The consumers read the slot through the generic proxy; the TMA boxes below write it
        // through the async proxy. The empty barrier orders those reads before this point, and
        // this cross-proxy fence orders them before the new boxes (without it, a warp's loads of
        // the slot's first rows could return the next stage's bytes, about one forward in 100).
        tc::fence_proxy_async_smem();
        unsigned char* st = smem + stage * kStageBytes;
        // weights and scales are read once per call: evict them from L2 first (made here, per
        // stage, so that the policy holds no register across the loop)
        const uint64_t pol = l2_evict_first_policy();
        if (lane == 0) {
          StageHdr* h = reinterpret_cast<StageHdr*>(st + kHdrOff);
          h->e = e; h->rbase = rbase; h->nvalid = nvalid; h->blk = blk; h->ks = 0; h->cidx = cidx;
          h->g = g; h->gbeg = gbeg; h->gend = gend; h->done = 0; h->split = split;
          tc::mbar_arrive_expect_tx(&full[stage], tx_bytes);
          tc::tma_load_2d_hint(st, &map0, g * 64, static_cast<int32_t>(wrow0), &full[stage], pol);
          if (kGateUp)
            tc::tma_load_2d_hint(st + kRB * 64, &map1, g * 64, static_cast<int32_t>(wrow0),
                                 &full[stage], pol);
          if (kScTma) {
            // the aligned run of 8 scale groups holding this stage's group(s): 16 bytes per row
            const int sx = (kG == 64 ? 2 * g : kG == 128 ? g : g >> 1) & ~7;
            tc::tma_load_2d_hint(st + kScOff, &smap0, sx, static_cast<int32_t>(wrow0),
                                 &full[stage], pol);
            if (kGateUp)
              tc::tma_load_2d_hint(st + kScOff + kRB * 16, &smap1, sx,
                                   static_cast<int32_t>(wrow0), &full[stage], pol);
          }
        }
        // scales: the 4-byte fp16 pair holding group g, 8 rows per lane
        // 4-byte scale pair holding this block's scale(s): groups 2g, 2g+1 (kG = 64), g (128) or
        // g / 2 (256), the pair starting at an even group
        const int gp = kG == 64 ? 2 * g : kG == 128 ? (g & ~1) : ((g >> 1) & ~1);
#pragma unroll
        for (int i = 0; i < (kScTma ? 0 : 8); ++i) {
          const int r = lane + 32 * i;  // stage scale row
          const __half* sbase;
          int64_t row;
          if (kGateUp) {
            sbase = r < kRB ? a.scales0 : a.scales1;
            row = wrow0 + (r < kRB ? r : r - kRB);
          } else {
            sbase = a.scales0;
            row = wrow0 + r;
          }
          const bool in = kGateUp ? true : (blk * kRB + r < a.N);
          cp_async4(tc::smem_u32(st + kScOff + r * 4), sbase + (in ? row : wrow0) * srow + gp, in,
                    pol);
        }
        if (g == gbeg) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = 2 * i + (lane >> 4);
            const bool live = n < nvalid;
            amask |= live ? 1u << i : 0u;
            int src = rbase + (live ? n : 0);
            if (a.perm) src = __ldg(a.perm + src);
            arow[i] = src;
          }
        }
        auto issue_act = [&](int gg, unsigned char* sst, uint64_t* bar) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = 2 * i + (lane >> 4);
            const uint32_t dst = tc::smem_u32(sst + kActOff + n * 256 + (act_swz<kG>(n, q) << 4));
            const __nv_bfloat16* src = a.act + static_cast<int64_t>(arow[i]) * a.K + gg * kBlockK;
            cp_async16s(dst, reinterpret_cast<const char*>(src) + q * 16, (amask >> i) & 1u);
          }
          cp_async_arrive_noinc(bar);
        };
        if (waited) {
          issue_act(g, st, &full[stage]);
        } else {
          // down, first piece: weights and scales of up to kStages groups go out before waiting
          // for gate/up (which writes h); their activation copies follow the wait
          ++npend;
          if (npend == kStages || g == gend - 1) {
            griddep_wait();
            waited = true;
            int s0 = stage - (npend - 1);
            if (s0 < 0) s0 += kStages;
            for (int j = 0; j < npend; ++j) {
              const int ss = (s0 + j) % kStages;
              issue_act(g - (npend - 1) + j, smem + ss * kStageBytes, &full[ss]);
            }
          }
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    }
    if (!waited) griddep_wait();
    if (ok && tc::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, status)) {
      if (lane == 0) reinterpret_cast<StageHdr*>(smem + stage * kStageBytes + kHdrOff)->done = 1;
      __syncwarp();
      tc::mbar_arrive(&full[stage]);      // 32 lane arrivals
      if (lane == 0) tc::mbar_arrive(&full[stage]);  // + the expect_tx slot
    }
    // leave no copy in flight into this CTA's shared memory
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    if (*abort_flag) {
      // outstanding TMA boxes land on their full barriers: wait (bounded) for the last stages
      for (int s = 0; s < kStages; ++s) tc::mbar_wait_drain(&full[s], 0), tc::mbar_wait_drain(&full[s], 1);
    }
    return;
  }

  // -------------------------------------------------------------------- consumer warps
  griddep_wait();  // outputs and split-K scratch follow the previous kernel
  const int gq = lane >> 2, t4 = lane & 3;
  const uint32_t a1032[4] = {0x64086408u, 0x64086408u, 0x64086408u, 0x64086408u};  // f16 1032
  const uint32_t a72[4] = {0x54805480u, 0x54805480u, 0x54805480u, 0x54805480u};    // f16 72
  const int mtile = kGateUp ? 16 : 32;
  int stage = 0;
  uint32_t phase = 0;
  float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
  while (true) {
    if (!tc::mbar_wait(&full[stage], phase, abort_flag, status)) break;
    const unsigned char* st = smem + stage * kStageBytes;
    const StageHdr hd = *reinterpret_cast<const StageHdr*>(st + kHdrOff);
    if (hd.done) break;
    // weights: tile 0 rows (gate: w*16.., down: w*32..), tile 1 (up rows w*16.. / down w*32+16..)
    const unsigned char* t0 = st + (kGateUp ? warp * 16 : warp * 32) * 64;
    const unsigned char* t1 = kGateUp ? t0 + p.RB * 64 : t0 + 16 * 64;
    // 16 bytes of codes per row: one piece of 16, or (64-wide groups) 8 from each 32-byte half
    auto ldw = [&](const unsigned char* row) {
      if (kG == 64) {
        const uint2 lo = *reinterpret_cast<const uint2*>(row + t4 * 8);
        const uint2 hi = *reinterpret_cast<const uint2*>(row + 32 + t4 * 8);
        return make_uint4(lo.x, lo.y, hi.x, hi.y);
      }
      return *reinterpret_cast<const uint4*>(row + t4 * 16);
    };
    const uint4 a0l = ldw(t0 + gq * 64);
    const uint4 a0h = ldw(t0 + (gq + 8) * 64);
    const uint4 a1l = ldw(t1 + gq * 64);
    const uint4 a1h = ldw(t1 + (gq + 8) * 64);
    uint32_t X[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int qq = act_piece<kG>(t4, c);
      const uint4 b = *reinterpret_cast<const uint4*>(st + kActOff + gq * 256 + (act_swz<kG>(gq, qq) << 4));
      X[4 * c] = b.x; X[4 * c + 1] = b.y; X[4 * c + 2] = b.z; X[4 * c + 3] = b.w;
    }
    // scale pairs of rows gq, gq+8 of both tiles
    const int sr0 = kGateUp ? warp * 16 + gq : warp * 32 + gq;
    const int sr1 = kGateUp ? p.RB + warp * 16 + gq : warp * 32 + 16 + gq;
    // TMA rows: 16 bytes, the pair's word inside the stage's aligned run of 8 groups
    constexpr int kScW = Lay::kScRowBytes / 4;
    const int gpair = kG == 64 ? 2 * hd.g : kG == 128 ? (hd.g & ~1) : ((hd.g >> 1) & ~1);
    const uint32_t* sc = reinterpret_cast<const uint32_t*>(st + kScOff) + (kScTma ? ((gpair & 7) >> 1) : 0);
    const uint32_t s0a = sc[sr0 * kScW], s0b = sc[(sr0 + 8) * kScW], s1a = sc[sr1 * kScW],
                   s1b = sc[(sr1 + 8) * kScW];
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&empty[stage]);
    if (++stage == kStages) { stage = 0; phase ^= 1u; }

    if (hd.g == hd.gbeg) {
#pragma unroll
      for (int c = 0; c < 4; ++c) { acc0[c] = 0.f; acc1[c] = 0.f; }
    }
    const uint32_t w0l[4] = {a0l.x, a0l.y, a0l.z, a0l.w}, w0h[4] = {a0h.x, a0h.y, a0h.z, a0h.w};
    const uint32_t w1l[4] = {a1l.x, a1l.y, a1l.z, a1l.w}, w1h[4] = {a1h.x, a1h.y, a1h.z, a1h.w};
    auto h2f = [](uint32_t v, int sh) {
      return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> sh)));
    };
    // one group's sums: tile 0, tile 1, and the offsets both carry (weights 1032 + q / 72 + q)
    float p0[4], p1[4], cr[4];
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    // acc += s * (P - C) for the rows' scales
    auto flush = [&](float sa0, float sb0, float sa1, float sb1) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc0[c] = fmaf(c < 2 ? sa0 : sb0, p0[c] - cr[c], acc0[c]);
        acc1[c] = fmaf(c < 2 ? sa1 : sb1, p1[c] - cr[c], acc1[c]);
      }
    };
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // X[4j..4j+3] = (x0,x4) (x2,x6) | (x1,x5) (x3,x7) of chunk j: low-plane pair, high-plane pair
      const uint32_t xl0 = X[4 * j], xl1 = X[4 * j + 1], xh0 = X[4 * j + 2], xh1 = X[4 * j + 3];
      // a group's first step starts its sums from zero (64-wide groups: steps 0 and 2)
      const bool first = kG == 64 ? (j == 0 || j == 2) : (j == 0);
      // (first is a constant once the loop is unrolled)
      auto mma_acc = [&](float (&d)[4], const uint32_t (&fa)[4], uint32_t b0, uint32_t b1) {
        if (first) mma_f16_16816(d, fa, b0, b1, zero);
        else mma_f16_16816(d, fa, b0, b1, d);
      };
      mma_acc(cr, a1032, xl0, xl1);
      mma_f16_16816(cr, a72, xh0, xh1, cr);
      {
        const uint32_t vl = w0l[j], vh = w0h[j], vl8 = vl >> 8, vh8 = vh >> 8;
        const uint32_t flo[4] = {nib_lo_f16(vl), nib_lo_f16(vh), nib_lo_f16(vl8), nib_lo_f16(vh8)};
        const uint32_t fhi[4] = {nib_hi_f16(vl), nib_hi_f16(vh), nib_hi_f16(vl8), nib_hi_f16(vh8)};
        mma_acc(p0, flo, xl0, xl1);
        mma_f16_16816(p0, fhi, xh0, xh1, p0);
      }
      {
        const uint32_t vl = w1l[j], vh = w1h[j], vl8 = vl >> 8, vh8 = vh >> 8;
        const uint32_t flo[4] = {nib_lo_f16(vl), nib_lo_f16(vh), nib_lo_f16(vl8), nib_lo_f16(vh8)};
        const uint32_t fhi[4] = {nib_hi_f16(vl), nib_hi_f16(vh), nib_hi_f16(vl8), nib_hi_f16(vh8)};
        mma_acc(p1, flo, xl0, xl1);
        mma_f16_16816(p1, fhi, xh0, xh1, p1);
      }
      if (kG == 64 && (j == 1 || j == 3)) {
        // 64-wide groups: j = 0, 1 are the block's first group (low half of the scale pair),
        // j = 2, 3 its second (high half)
        const int sh = j == 1 ? 0 : 16;
        flush(h2f(s0a, sh), h2f(s0b, sh), h2f(s1a, sh), h2f(s1b, sh));
      }
    }
    if (kG != 64) {
      // the block's group is the low half of its pair for an even group index, the high half else
      const int sh = ((kG == 128 ? hd.g : hd.g >> 1) & 1) * 16;
      flush(h2f(s0a, sh), h2f(s0b, sh), h2f(s1a, sh), h2f(s1b, sh));
    }
    if (hd.g != hd.gend - 1) continue;

    // ------------------------------------------------------------------ item epilogue
    const int mt = hd.blk * kCW + warp;  // global tile index of this warp inside the expert
    if (mt * mtile >= a.N) continue;     // rows past the expert (last, partial block)
    bool write = true;
    if constexpr (kEven) {
      const int np = split_np(hd.split);
      if (np > 1) {
        // split tile: publish this piece's partial sums; the last piece to arrive reduces them
        const int tile = (hd.cidx * p.nblk + hd.blk) * kCW + warp;
        const int slot = 2 * static_cast<int>(blockIdx.x) + ((hd.split >> 24) & 1);
        float* part = a.split_part + (static_cast<int64_t>(slot) * kCW + warp) * 256 + lane * 8;
        reinterpret_cast<float4*>(part)[0] = make_float4(acc0[0], acc0[1], acc0[2], acc0[3]);
        reinterpret_cast<float4*>(part)[1] = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          last = (atomicAdd(a.split_cnt + tile, 1) == np - 1);
          if (last) a.split_cnt[tile] = 0;  // ready for the next launch that uses the scratch
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        write = last != 0;
        if (last) {
          __threadfence();
#pragma unroll
          for (int c = 0; c < 4; ++c) { acc0[c] = 0.f; acc1[c] = 0.f; }
          for (int pc = 0; pc < np; ++pc) {  // piece order: deterministic
            const float* src = a.split_part +
                               (static_cast<int64_t>(split_slot(hd.split, pc)) * kCW + warp) * 256 +
                               lane * 8;
            const float4 u = __ldcg(reinterpret_cast<const float4*>(src));
            const float4 v = __ldcg(reinterpret_cast<const float4*>(src) + 1);
            acc0[0] += u.x; acc0[1] += u.y; acc0[2] += u.z; acc0[3] += u.w;
            acc1[0] += v.x; acc1[1] += v.y; acc1[2] += v.z; acc1[3] += v.w;
          }
        }
      }
    } else if (KS > 1) {
      // split-K: publish this split's partial sums; the last split to arrive reduces them
      const int tile = (hd.cidx * p.nblk + hd.blk) * kCW + warp;
      float* part = a.split_part + (static_cast<int64_t>(tile) * KS + hd.ks) * 256 + lane * 8;
      reinterpret_cast<float4*>(part)[0] = make_float4(acc0[0], acc0[1], acc0[2], acc0[3]);
      reinterpret_cast<float4*>(part)[1] = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        last = (atomicAdd(a.split_cnt + tile, 1) == KS - 1);
        if (last) a.split_cnt[tile] = 0;  // ready for the next launch that uses the scratch
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      write = last != 0;
      if (last) {
        __threadfence();
        const float* base = a.split_part + static_cast<int64_t>(tile) * KS * 256 + lane * 8;
#pragma unroll
        for (int c = 0; c < 4; ++c) { acc0[c] = 0.f; acc1[c] = 0.f; }
        for (int s = 0; s < KS; ++s) {  // split order: deterministic
          const float4 u = __ldcg(reinterpret_cast<const float4*>(base + s * 256));
          const float4 v = __ldcg(reinterpret_cast<const float4*>(base + s * 256) + 1);
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
        if (col >= hd.nvalid) continue;
        const int64_t orow = hd.rbase + col;
        // the activation row was stored times 2^-e: the sums are at that scale
        const int e = a.aexp ? a.aexp[a.perm ? a.perm[orow] : orow] : 0;
        if (kGateUp) {
          // h columns: element i of every 8 at position bitrev3(i) (the down GEMM's B order), as
          // f16, stored times 2^-2e (u and v are at scale 2^-e each)
          const int n0 = mt * 16 + (((gq & 1) << 2) | (gq & 2) | (gq >> 2));
          __half* hrow = static_cast<__half*>(a.out) + orow * a.N;
          const float up = exp2i(e);
          hrow[n0] = f32_to_f16_sat(silu_scaled(acc0[c], up) * acc1[c]);
          hrow[n0 + 8] = f32_to_f16_sat(silu_scaled(acc0[c + 2], up) * acc1[c + 2]);
          if (a.hexp && mt == 0 && gq == 0) a.hexp[orow] = 2 * e;
        } else {
          const int n0 = mt * 32 + gq;
          const float up = exp2i(e);
          float* y = static_cast<float*>(a.out) + orow * a.N;
          y[n0] = acc0[c] * up;
          y[n0 + 8] = acc0[c + 2] * up;
          y[n0 + 16] = acc1[c] * up;
          y[n0 + 24] = acc1[c + 2] * up;
        }
      }
    }
  }
}

// Codes [rows, K/2] bytes: boxes of 64 bytes (one group) x box_rows rows, no swizzle, zero fill.
static PFN_cuTensorMapEncodeTiled_v12000 cta_tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}
static bool make_codes_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t K,
                            int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = cta_tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scales [rows, groups] fp16: boxes of 8 groups (16 bytes) x box_rows rows, zero fill. Needs a
// 16-byte aligned base and a row stride that is a multiple of 16 bytes.
static bool make_scales_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t groups,
                             int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = cta_tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(groups), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(groups) * 2};
  cuuint32_t box[2] = {8, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kGateUp, int kG, bool kScTma, bool kEven>
cudaError_t launch_t(const GemmArgs& a, int64_t experts, int num_sms, cudaStream_t stream) {
  // the kEven split words hold CTA indices and piece counts in 12 bits
  if (kEven && (num_sms < 1 || num_sms * kCtasPerSm > 4096)) return cudaErrorInvalidValue;
  CtaGemmParams p;
  p.a = a;
  p.RB = cta_gemm_block_rows(kGateUp);
  p.nblk = static_cast<int>((a.N + p.RB - 1) / p.RB);
  CUtensorMap m0, m1, s0, s1;
  const int64_t rows = experts * a.N;
  if (!make_codes_tmap(&m0, a.codes0, rows, a.K, p.RB)) return cudaErrorInvalidValue;
  if (!make_codes_tmap(&m1, kGateUp ? a.codes1 : a.codes0, rows, a.K, p.RB))
    return cudaErrorInvalidValue;
  if (kScTma) {
    if (!make_scales_tmap(&s0, a.scales0, rows, a.K / kG, p.RB)) return cudaErrorInvalidValue;
    if (!make_scales_tmap(&s1, kGateUp ? a.scales1 : a.scales0, rows, a.K / kG, p.RB))
      return cudaErrorInvalidValue;
  } else {
    s0 = m0;  // not read
    s1 = m1;
  }
  auto kern = grouped_gemm_cta_kernel<kGateUp, kG, kScTma, kEven>;
  constexpr int smem = CtaLayout<kScTma>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)  // two CTAs per SM need (nearly) all of its shared memory
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(num_sms * kCtasPerSm), dim3(kThreads), smem, stream, true, m0,
                       m1, s0, s1, p);
}

// The TMA scale path when every scale row starts on a 16-byte boundary.
template <bool kGateUp, int kG>
cudaError_t launch_g(const GemmArgs& a, int64_t experts, int num_sms, bool even,
                     cudaStream_t stream) {
  const int64_t row_bytes = static_cast<int64_t>(a.K / kG) * 2;
  const bool tma = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(a.scales0) % 16 == 0 &&
                   (!kGateUp || reinterpret_cast<uintptr_t>(a.scales1) % 16 == 0);
  if (even)
    return tma ? launch_t<kGateUp, kG, true, true>(a, experts, num_sms, stream)
               : launch_t<kGateUp, kG, false, true>(a, experts, num_sms, stream);
  return tma ? launch_t<kGateUp, kG, true, false>(a, experts, num_sms, stream)
             : launch_t<kGateUp, kG, false, false>(a, experts, num_sms, stream);
}

}  // namespace

int cta_gemm_block_rows(bool gate_up) { return gate_up ? kCW * 16 : kCW * 32; }
int cta_gemm_warps() { return kCW; }

cudaError_t launch_gemm_cta(const GemmArgs& a, bool gate_up, int64_t experts, int num_sms,
                            bool even, cudaStream_t stream) {
  switch (a.group) {
    case 64:
      return gate_up ? launch_g<true, 64>(a, experts, num_sms, even, stream)
                     : launch_g<false, 64>(a, experts, num_sms, even, stream);
    case 256:
      return gate_up ? launch_g<true, 256>(a, experts, num_sms, even, stream)
                     : launch_g<false, 256>(a, experts, num_sms, even, stream);
    default:
      return gate_up ? launch_g<true, 128>(a, experts, num_sms, even, stream)
                     : launch_g<false, 128>(a, experts, num_sms, even, stream);
  }
}

// The kEven schedule for a launch with at most max_tiles (chunk x row block) tiles: when even
// that many leave at most two tiles per CTA (the count is an upper bound: experts that several
// tokens share make fewer chunks).
bool cta_gemm_even(int64_t max_tiles, int num_sms) {
  return max_tiles <= 2 * static_cast<int64_t>(num_sms) * kCtasPerSm;
}

// kEven partial-sum scratch of a launch on num_sms SMs: two slots per CTA (its range's first and
// last piece), 256 floats per consumer warp each.
int64_t cta_gemm_partial_floats(int num_sms) {
  return static_cast<int64_t>(2) * num_sms * kCtasPerSm * kCW * 256;
}

// Contraction splits for a batch whose grouped GEMM has `items` (chunk x row block) work items:
// enough for about two items per CTA, each split keeping at least two 128-wide groups.
// Contraction splits per work item. An item streams K/128 stages of 16 KB; a split piece also
// pays the cross-CTA reduction of its partial sums (a fence, an atomic and the loads of the other
// splits' partials: about 3.5 stages' time, measured at the decode shapes). The persistent CTAs
// take the pieces in rounds, so ks splits cost about rounds(ks) x (stages per piece + reduction),
// rounds = ceil(items * ks / CTAs). Only counts that give every CTA a piece in the first round are
// weighed (a CTA's stream rate is capped by its consumers, so idle CTAs lose bandwidth), unless no
// count reaches that; the cheapest wins (the fewest splits on a tie), and a piece keeps at least
// 2 stages.
int cta_gemm_ksplit(int64_t items, int64_t K, int num_sms) {
  const int64_t ctas = static_cast<int64_t>(num_sms) * kCtasPerSm;
  const int64_t groups = K / kBlockK;
  constexpr double kReduceStages = 3.5;
  int ks_max = 1;
  while (2 * ks_max <= 16 && groups >= 2 * (2 * ks_max)) ks_max *= 2;
  int best = 0;
  double best_cost = 0.0;
  for (int ks = 1; ks <= ks_max; ks *= 2) {
    if (items * ks < ctas && ks < ks_max) continue;  // leaves CTAs idle in the first round
    const int64_t rounds = (items * ks + ctas - 1) / ctas;
    const double cost = static_cast<double>(rounds) *
                        (static_cast<double>(groups) / ks + (ks > 1 ? kReduceStages : 0.0));
    if (best == 0 || cost < best_cost) {
      best_cost = cost;
      best = ks;
    }
  }
  return best;
}

}  // namespace strata
