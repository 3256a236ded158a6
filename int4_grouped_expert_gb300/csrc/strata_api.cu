// The C ABI (include/strata.h): host-side argument checks, workspace layout and the launch
// sequence of one MoE layer. Nothing here allocates device memory; every check runs before the
// first CUDA call of an entry point.
#include <cstdint>
#include <cstring>

#include <algorithm>

#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace strata {

constexpr int64_t kMaxTokens = int64_t(1) << 22;
constexpr int64_t kMaxDim = int64_t(1) << 16;
constexpr int kRouterSplitsForSizing = 256;  // SM count bound used to size the router scratch
constexpr size_t kAlign = 256;

static size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct RouteLayout {
  size_t hdr, partial, ids, gates, counts, offsets, perm, inv, total;
};
static RouteLayout route_layout(int64_t T, int64_t H, int E, int k, int shared, size_t base = 0) {
  RouteLayout L{};
  size_t o = base;
  const int ns = router_num_splits(T, H, E, kRouterSplitsForSizing);
  const int64_t R = T * k;
  L.hdr = o; o = up(o + sizeof(WsHeader));
  const size_t pf = static_cast<size_t>(ns) * T * E;  // >= T * E: also the decode logits
  L.partial = o; o = up(o + sizeof(float) * pf);
  L.ids = o; o = up(o + sizeof(int) * R);
  L.gates = o; o = up(o + sizeof(float) * R);
  L.counts = o; o = up(o + sizeof(int) * (E + 1));
  L.offsets = o; o = up(o + sizeof(int) * (E + 2));
  L.perm = o; o = up(o + sizeof(int) * (R + shared * T));
  L.inv = o; o = up(o + sizeof(int) * R);
  L.total = o;
  return L;
}

struct FwdLayout {
  RouteLayout r;
  size_t seg_expert, seg_row0, seg_rows, seg_item_gu, seg_item_dn, chunk_list, h, y, xp,
      xexp, rexp, hexp, split_part, split_cnt, total;
  int ksplit;     // gate/up contraction splits (warp paths)
  int ksplit_dn;  // down contraction splits (CTA-staged warp path)
  int nblk_gu, nblk_dn;  // CTA-staged warp path: row blocks per expert
  bool even_gu, even_dn; // CTA-staged warp path: equal stage ranges per CTA (smallest batches)
  bool tc;   // tensor-core path for the grouped GEMMs
  bool cta;  // CTA-staged warp GEMM (else the per-warp one)
};

#ifndef STRATA_WARP_GEMM_LEGACY
#define STRATA_WARP_GEMM_LEGACY 0
#endif
// SM count the work split is sized for (the same on every device, so the workspace size and the
// launch agree): it steers how many contraction splits small batches get and which take equal
// stage ranges, whose partial-sum scratch is sized for at most this many SMs.
constexpr int kSizingSms = 152;

// Tensor-core path for batches with enough rows per expert to fill 128 x N tiles, and for layers
// with 8-bit codes at every batch size (the warp kernels read 4-bit codes only).
static bool use_tc_path(const strata_moe_layer* L, int64_t T) {
  if (L->bits == 8) return true;
  if (L->flags & STRATA_FORCE_WARP_PATH) return false;
  if (L->flags & STRATA_FORCE_TC_PATH) return true;
  return T >= 128;
}
// Token rows per tensor-core tile: 64 when the routed experts average at most 48 rows (the
// small-tile kernel streams its code tiles through a deep TMA ring) or the codes are 8-bit (they
// go through that ring only), else 256.
static int tc_tile_rows(const strata_moe_layer* L, int64_t T) {
  if (L->bits == 8) return kTcRowsSmall;
  return T * L->k <= 48 * static_cast<int64_t>(L->E) ? kTcRowsSmall : kTcRows;
}
static int layer_group(const strata_moe_layer* L) {
  return L->group_size == 0 ? STRATA_GROUP : L->group_size;
}
static int layer_bits(const strata_moe_layer* L) { return L->bits == 0 ? 4 : L->bits; }

static FwdLayout fwd_layout(const strata_moe_layer* L, int64_t T) {
  FwdLayout F{};
  F.r = route_layout(T, L->H, L->E, L->k, L->has_shared);
  size_t o = F.r.total;
  const int nseg = L->E + 2;
  const int64_t rows = T * L->k + (L->has_shared ? T : 0);
  F.seg_expert = o; o = up(o + sizeof(int) * nseg);
  F.seg_row0 = o; o = up(o + sizeof(int) * nseg);
  F.seg_rows = o; o = up(o + sizeof(int) * nseg);
  F.seg_item_gu = o; o = up(o + sizeof(int) * nseg);
  F.seg_item_dn = o; o = up(o + sizeof(int) * nseg);
  F.tc = use_tc_path(L, T);
  const int64_t segs = (T * L->k < L->E ? T * L->k : L->E) + L->has_shared;
  const int64_t max_chunks = rows / 8 + segs;  // 8-row chunks of the warp path
  F.chunk_list = o; o = up(o + sizeof(int4) * (F.tc ? 0 : max_chunks));
  F.h = o; o = up(o + sizeof(uint16_t) * rows * L->I);
  F.y = o; o = up(o + sizeof(float) * rows * L->H);
  F.xp = o; o = up(o + sizeof(uint16_t) * rows * L->H);  // gathered / pair-interleaved x
  // range exponents of the f16 GEMM operands: per token of x_perm, per gathered row, per h row
  F.xexp = o; o = up(o + sizeof(int) * T);
  F.rexp = o; o = up(o + sizeof(int) * rows);
  F.hexp = o; o = up(o + sizeof(int) * rows);
  // the CTA-staged kernel reads scale pairs with 4-byte copies: even group counts only
  // (256-wide groups: the pair holding a block's scale starts at an even group: K / 256 even)
  const int G = layer_group(L);
  F.cta = !F.tc && !STRATA_WARP_GEMM_LEGACY && (L->H / 128) % 2 == 0 && (L->I / 128) % 2 == 0 &&
          (G != 256 || ((L->H / 256) % 2 == 0 && (L->I / 256) % 2 == 0)) &&
          aligned(L->gate_scales, 4) && aligned(L->up_scales, 4) && aligned(L->down_scales, 4);
  F.ksplit = 1;
  F.ksplit_dn = 1;
  F.even_gu = F.even_dn = false;
  int64_t part_floats = 0, ncnt = 0;
  if (F.cta) {
    F.nblk_gu = static_cast<int>((L->I + cta_gemm_block_rows(true) - 1) / cta_gemm_block_rows(true));
    F.nblk_dn = static_cast<int>((L->H + cta_gemm_block_rows(false) - 1) / cta_gemm_block_rows(false));
    // batches that leave at most two tiles per CTA take equal stage ranges, the others whole
    // tiles with contraction splits
    F.even_gu = cta_gemm_even(max_chunks * F.nblk_gu, kSizingSms);
    F.even_dn = cta_gemm_even(max_chunks * F.nblk_dn, kSizingSms);
    if (!F.even_gu) F.ksplit = cta_gemm_ksplit(segs * F.nblk_gu, L->H, kSizingSms);
    if (!F.even_dn) F.ksplit_dn = cta_gemm_ksplit(segs * F.nblk_dn, L->I, kSizingSms);
    // per split tile: one arrival counter per consumer warp; split-K: one 256-float partial per
    // split too; equal ranges: two slots per CTA
    const bool cnt_gu = F.ksplit > 1 || F.even_gu, cnt_dn = F.ksplit_dn > 1 || F.even_dn;
    const int64_t tgu = cnt_gu ? max_chunks * F.nblk_gu * cta_gemm_warps() : 0;
    const int64_t tdn = cnt_dn ? max_chunks * F.nblk_dn * cta_gemm_warps() : 0;
    part_floats = std::max((F.ksplit > 1 ? tgu * F.ksplit : 0), (F.ksplit_dn > 1 ? tdn * F.ksplit_dn : 0)) * 256;
    if (F.even_gu || F.even_dn) part_floats = std::max(part_floats, cta_gemm_partial_floats(kSizingSms));
    ncnt = std::max(tgu, tdn);
  } else if (!F.tc) {
    F.ksplit = warp_ksplit(T, L->E, L->k, L->has_shared, L->I, L->H);
    // split-K scratch: tiles <= chunks * (I / 16)
    ncnt = F.ksplit > 1 ? max_chunks * (L->I / 16) : 0;
    part_floats = 256 * F.ksplit * ncnt;
  }
  F.split_part = o; o = up(o + sizeof(float) * part_floats);
  F.split_cnt = o; o = up(o + sizeof(int) * ncnt);
  F.total = o;
  return F;
}

static strata_status cuda_fail(cudaError_t e) {
  return e == cudaSuccess ? STRATA_OK : STRATA_ERR_CUDA;
}

static int device_sms(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return 0;
}

static strata_status check_layer(const strata_moe_layer* L) {
  if (!L) return STRATA_ERR_INVALID_ARG;
  if (L->H <= 0 || L->I <= 0 || L->H > kMaxDim || L->I > kMaxDim) return STRATA_ERR_SHAPE;
  const int G = layer_group(L);
  if (G != 64 && G != 128 && G != 256) return STRATA_ERR_UNSUPPORTED;
  if (layer_bits(L) != 4 && layer_bits(L) != 8) return STRATA_ERR_UNSUPPORTED;
  if (L->H % STRATA_GROUP || L->I % STRATA_GROUP || L->H % G || L->I % G) return STRATA_ERR_SHAPE;
  if (L->has_shared != 0 && L->has_shared != 1) return STRATA_ERR_INVALID_ARG;
  if (L->E < 1 || L->E + L->has_shared > STRATA_MAX_EXPERTS) return STRATA_ERR_UNSUPPORTED;
  if (L->k < 1 || L->k > L->E || L->k > STRATA_MAX_TOPK) return STRATA_ERR_INVALID_ARG;
  if (L->flags & ~(STRATA_RENORM | STRATA_ADD_RESIDUAL | STRATA_ROUTER_FP16 | STRATA_FORCE_WARP_PATH |
                   STRATA_FORCE_TC_PATH | STRATA_WS_REUSE))
    return STRATA_ERR_INVALID_ARG;
  if ((L->flags & STRATA_FORCE_WARP_PATH) && (L->flags & STRATA_FORCE_TC_PATH))
    return STRATA_ERR_INVALID_ARG;
  if (!L->w_router || !L->gate_codes || !L->gate_scales || !L->up_codes || !L->up_scales ||
      !L->down_codes || !L->down_scales)
    return STRATA_ERR_INVALID_ARG;
  if (!aligned(L->w_router, 16) || !aligned(L->gate_codes, 16) || !aligned(L->up_codes, 16) ||
      !aligned(L->down_codes, 16) || !aligned(L->gate_scales, 2) || !aligned(L->up_scales, 2) ||
      !aligned(L->down_scales, 2) || (L->bias && !aligned(L->bias, 4)))
    return STRATA_ERR_INVALID_ARG;
  return STRATA_OK;
}

struct Taps {
  int32_t* ids;
  float* gates;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
};

static strata_status run_forward(const strata_moe_layer* L, const void* x, int64_t T, void* out,
                                 const Taps* taps, void* ws, size_t ws_bytes, cudaStream_t st,
                                 void* const* events = nullptr, bool keep_status = false,
                                 unsigned long long* hits = nullptr,
                                 const int32_t* T_dev = nullptr) {
  auto mark = [&](int i) -> bool {
    if (!events || !events[i]) return true;
    return cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) == cudaSuccess;
  };
  strata_status s = check_layer(L);
  if (s != STRATA_OK) return s;
  if (T < 0 || T > kMaxTokens) return STRATA_ERR_SHAPE;
  if (T == 0) return STRATA_OK;
  if (!x || !out) return STRATA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16)) return STRATA_ERR_INVALID_ARG;
  if (x == out) return STRATA_ERR_INVALID_ARG;
  const FwdLayout F = fwd_layout(L, T);
  // the per-warp decode kernel (odd group counts, 2-byte-aligned scales) has 128-wide groups only
  if (!F.tc && !F.cta && layer_group(L) != STRATA_GROUP) return STRATA_ERR_UNSUPPORTED;
  // 8-bit codes run on the tensor-core kernel, which a forced warp path would bypass
  if (layer_bits(L) == 8 && (L->flags & STRATA_FORCE_WARP_PATH)) return STRATA_ERR_UNSUPPORTED;
  // a device token count needs the fused decode router and the decode GEMMs (whose work lists
  // are built on the device): T is then the maximum batch
  if (T_dev && (T > kRouteSmallMaxT || F.tc || taps)) return STRATA_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, kAlign)) return STRATA_ERR_WORKSPACE;
  if (ws_bytes < F.total) return STRATA_ERR_WORKSPACE;

  int sms = 0;
  if (device_sms(&sms) != 0) return STRATA_ERR_CUDA;
  char* base = static_cast<char*>(ws);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(base + F.r.hdr);
  const int E = L->E, k = L->k, S = L->has_shared;
  const int64_t R = T * k;
  int* ids = reinterpret_cast<int*>(base + F.r.ids);
  float* gates = reinterpret_cast<float*>(base + F.r.gates);
  int* counts = reinterpret_cast<int*>(base + F.r.counts);
  int* offsets = reinterpret_cast<int*>(base + F.r.offsets);
  int* perm = reinterpret_cast<int*>(base + F.r.perm);
  int* inv = reinterpret_cast<int*>(base + F.r.inv);

  if (!mark(0)) return STRATA_ERR_CUDA;
  // keep_status: a later layer of a stack clears the counters but keeps the status word, so a
  // fault flagged by any layer stays visible after the whole stack. STRATA_WS_REUSE: the header
  // is zero or as the last completed call left it (the fused router resets its counters as it
  // ends), so no clearing op runs between the previous kernel and this call's first one.
  cudaError_t e = cudaSuccess;
  if (!(L->flags & STRATA_WS_REUSE)) {
    const size_t clear_from = keep_status ? sizeof(hdr->status) : 0;
    e = cudaMemsetAsync(reinterpret_cast<char*>(hdr) + clear_from, 0,
                        sizeof(WsHeader) - clear_from, st);
    if (e != cudaSuccess) return STRATA_ERR_CUDA;
  }

  PermuteArgs pa{};
  pa.ids = ids;
  pa.T = static_cast<int>(T);
  pa.k = k;
  pa.E = E;
  pa.has_shared = S;
  pa.counts = counts;
  pa.offsets = offsets;
  pa.perm = perm;
  pa.inv = inv;
  pa.seg_expert = reinterpret_cast<int*>(base + F.seg_expert);
  pa.seg_row0 = reinterpret_cast<int*>(base + F.seg_row0);
  pa.seg_rows = reinterpret_cast<int*>(base + F.seg_rows);
  pa.seg_item_gu = reinterpret_cast<int*>(base + F.seg_item_gu);
  pa.seg_item_dn = reinterpret_cast<int*>(base + F.seg_item_dn);
  pa.ksplit_dn = 1;
  pa.cnt_per_chunk = 0;
  if (F.tc) {
    pa.tokc = tc_tile_rows(L, T);
    pa.mtiles_gu = static_cast<int>(L->I / 128);
    pa.mtiles_dn = static_cast<int>(L->H / 128);
    pa.ksplit_gu = 1;
    pa.chunk_list = nullptr;
  } else if (F.cta) {
    pa.tokc = 8;
    pa.mtiles_gu = F.nblk_gu;
    pa.mtiles_dn = F.nblk_dn;
    pa.ksplit_gu = F.ksplit;
    pa.ksplit_dn = F.ksplit_dn;
    pa.cnt_per_chunk = (F.ksplit > 1 || F.ksplit_dn > 1 || F.even_gu || F.even_dn)
                           ? std::max(F.nblk_gu, F.nblk_dn) * cta_gemm_warps() : 0;
    pa.chunk_list = reinterpret_cast<int4*>(base + F.chunk_list);
  } else {
    pa.tokc = 8;
    pa.mtiles_gu = static_cast<int>(L->I / 16);
    pa.mtiles_dn = static_cast<int>(L->H / 32);
    pa.ksplit_gu = F.ksplit;
    pa.cnt_per_chunk = F.ksplit > 1 ? pa.mtiles_gu : 0;
    pa.chunk_list = reinterpret_cast<int4*>(base + F.chunk_list);
  }
  pa.split_cnt = pa.cnt_per_chunk > 0 ? reinterpret_cast<int*>(base + F.split_cnt) : nullptr;
  pa.hits = hits;
  pa.hdr = hdr;
  pa.status = &hdr->status;

  if (T <= kRouteSmallMaxT) {
    RouteSmallArgs ra{};
    ra.x = static_cast<const __nv_bfloat16*>(x);
    ra.wr = L->w_router;
    ra.wr_fp16 = (L->flags & STRATA_ROUTER_FP16) != 0;
    ra.bias = L->bias;
    ra.T = static_cast<int>(T);
    ra.T_dev = T_dev;
    ra.H = static_cast<int>(L->H);
    ra.E = E;
    ra.k = k;
    ra.flags = L->flags & STRATA_RENORM;
    ra.epc = route_small_epc(E, sms);
    ra.logits = reinterpret_cast<float*>(base + F.r.partial);
    ra.ids = ids;
    ra.gates = gates;
    ra.x_perm = F.tc ? nullptr : base + F.xp;
    ra.x_f16 = F.cta;  // the CTA-staged GEMM multiplies f16 operands
    ra.xexp = reinterpret_cast<int*>(base + F.xexp);
    ra.grp = pa;
    ra.do_group = true;
    e = launch_route_small(ra, st);
    if (e != cudaSuccess || !mark(1) || !mark(2)) return STRATA_ERR_CUDA;
  } else {
    const int nsplit = router_num_splits(T, L->H, E, sms);
    e = launch_router(x, L->w_router, L->bias, T, L->H, E, k,
                      L->flags & (STRATA_RENORM | STRATA_ROUTER_FP16), nsplit,
                      reinterpret_cast<float*>(base + F.r.partial), ids, gates, st);
    if (e != cudaSuccess || !mark(1)) return STRATA_ERR_CUDA;
    e = launch_permute(pa, st);
    if (e != cudaSuccess || !mark(2)) return STRATA_ERR_CUDA;
  }

  const int64_t rows = R + (S ? T : 0);
  if (F.tc) {
    e = launch_gather_rows(x, perm, rows, L->H, base + F.xp, kGatherTc,
                           reinterpret_cast<int*>(base + F.rexp), st);
    if (e != cudaSuccess) return STRATA_ERR_CUDA;
    TcArgs g{};
    g.group = layer_group(L);
    g.bits = layer_bits(L);
    g.codes0 = L->gate_codes;
    g.scales0 = static_cast<const __half*>(L->gate_scales);
    g.codes1 = L->up_codes;
    g.scales1 = static_cast<const __half*>(L->up_scales);
    g.out = base + F.h;
    g.K = static_cast<int>(L->H);
    g.Nw = static_cast<int>(L->I);
    g.hdr = hdr;
    g.aexp = reinterpret_cast<const int*>(base + F.rexp);
    g.hexp = reinterpret_cast<int*>(base + F.hexp);
    g.seg_expert = pa.seg_expert;
    g.seg_row0 = pa.seg_row0;
    g.seg_rows = pa.seg_rows;
    g.seg_item = pa.seg_item_gu;
    g.status = &hdr->status;
    const int64_t nexp = E + (S ? 1 : 0);
    e = launch_gemm_tc(g, true, base + F.xp, rows, nexp, pa.tokc, sms, st);
    if (e != cudaSuccess || !mark(3)) return STRATA_ERR_CUDA;
    TcArgs d = g;
    d.codes0 = L->down_codes;
    d.scales0 = static_cast<const __half*>(L->down_scales);
    d.codes1 = nullptr;
    d.scales1 = nullptr;
    d.out = base + F.y;
    d.K = static_cast<int>(L->I);
    d.Nw = static_cast<int>(L->H);
    d.aexp = g.hexp;
    d.hexp = nullptr;
    d.seg_item = pa.seg_item_dn;
    e = launch_gemm_tc(d, false, base + F.h, rows, nexp, pa.tokc, sms, st);
    if (e != cudaSuccess || !mark(4)) return STRATA_ERR_CUDA;
  } else {
    GemmArgs g{};
    g.group = layer_group(L);
    g.codes0 = L->gate_codes;
    g.scales0 = static_cast<const __half*>(L->gate_scales);
    g.codes1 = L->up_codes;
    g.scales1 = static_cast<const __half*>(L->up_scales);
    g.act = reinterpret_cast<const __nv_bfloat16*>(base + F.xp);
    if (T <= kRouteSmallMaxT) {
      g.perm = perm;  // x_perm rows are tokens
      g.aexp = F.cta ? reinterpret_cast<const int*>(base + F.xexp) : nullptr;
    } else {
      e = launch_gather_rows(x, perm, rows, L->H, base + F.xp, F.cta ? kGatherCta : kGatherWarp,
                             F.cta ? reinterpret_cast<int*>(base + F.rexp) : nullptr, st);
      if (e != cudaSuccess) return STRATA_ERR_CUDA;
      g.perm = nullptr;  // xp rows are GEMM rows
      g.aexp = F.cta ? reinterpret_cast<const int*>(base + F.rexp) : nullptr;
    }
    g.hexp = F.cta ? reinterpret_cast<int*>(base + F.hexp) : nullptr;
    g.out = base + F.h;
    g.K = static_cast<int>(L->H);
    g.N = static_cast<int>(L->I);
    g.hdr = hdr;
    g.chunk_list = pa.chunk_list;
    g.ksplit = F.ksplit;
    g.split_part = reinterpret_cast<float*>(base + F.split_part);
    g.split_cnt = pa.split_cnt;
    const int64_t experts = E + S;
    // the equal-range schedule's scratch is sized for at most kSizingSms SMs
    e = F.cta ? launch_gemm_cta(g, true, experts, F.even_gu ? std::min(sms, kSizingSms) : sms,
                                F.even_gu, st)
              : launch_gemm_warp(g, true, sms, st);
    if (e != cudaSuccess || !mark(3)) return STRATA_ERR_CUDA;
    GemmArgs d = g;
    d.codes0 = L->down_codes;
    d.scales0 = static_cast<const __half*>(L->down_scales);
    d.codes1 = nullptr;
    d.scales1 = nullptr;
    d.act = reinterpret_cast<const __nv_bfloat16*>(base + F.h);
    d.perm = nullptr;
    d.aexp = g.hexp;
    d.hexp = nullptr;
    d.out = base + F.y;
    d.K = static_cast<int>(L->I);
    d.N = static_cast<int>(L->H);
    d.ksplit = F.cta ? F.ksplit_dn : 1;
    e = F.cta ? launch_gemm_cta(d, false, experts, F.even_dn ? std::min(sms, kSizingSms) : sms,
                                F.even_dn, st)
              : launch_gemm_warp(d, false, sms, st);
    if (e != cudaSuccess || !mark(4)) return STRATA_ERR_CUDA;
  }

  e = launch_combine(reinterpret_cast<const float*>(base + F.y), gates, inv, x, T, L->H, k, S, R,
                     (L->flags & STRATA_ADD_RESIDUAL) ? 1 : 0, out, T_dev, st);
  if (e != cudaSuccess || !mark(5)) return STRATA_ERR_CUDA;

  if (taps) {
    struct { void* dst; const void* src; size_t n; } cp[] = {
        {taps->ids, ids, sizeof(int) * R},           {taps->gates, gates, sizeof(float) * R},
        {taps->counts, counts, sizeof(int) * E},     {taps->offsets, offsets, sizeof(int) * (E + 1)},
        {taps->perm, perm, sizeof(int) * R},         {taps->inv, inv, sizeof(int) * R}};
    for (auto& c : cp)
      if (c.dst && cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return STRATA_ERR_CUDA;
  }
  return STRATA_OK;
}

// Argument checks of the router entry points (strata_route_topk and its no-workspace variant),
// in the order both apply them.
strata_status check_route_args(const void* x_bf16, const void* w_router, int64_t T, int64_t H,
                               int32_t E, int32_t k, uint32_t flags, const int32_t* ids,
                               const float* gates, const int32_t* counts, const int32_t* offsets,
                               const int32_t* perm, const int32_t* inv) {
  if (T < 0 || T > kMaxTokens || H <= 0 || H > kMaxDim || H % STRATA_GROUP) return STRATA_ERR_SHAPE;
  if (E < 1 || E > STRATA_MAX_EXPERTS) return STRATA_ERR_UNSUPPORTED;
  if (k < 1 || k > E || k > STRATA_MAX_TOPK) return STRATA_ERR_INVALID_ARG;
  if (flags & ~(STRATA_RENORM | STRATA_ROUTER_FP16)) return STRATA_ERR_INVALID_ARG;
  const bool any_group = counts || offsets || perm || inv;
  const bool all_group = counts && offsets && perm && inv;
  if (any_group && !all_group) return STRATA_ERR_INVALID_ARG;
  if (T > 0 && (!x_bf16 || !w_router || !ids || !gates)) return STRATA_ERR_INVALID_ARG;
  if ((x_bf16 && !aligned(x_bf16, 16)) || (w_router && !aligned(w_router, 16)))
    return STRATA_ERR_INVALID_ARG;
  return STRATA_OK;
}

}  // namespace strata

using namespace strata;

extern "C" {

const char* strata_status_string(int status) {
  switch (status) {
    case STRATA_OK: return "STRATA_OK";
    case STRATA_ERR_INVALID_ARG: return "STRATA_ERR_INVALID_ARG";
    case STRATA_ERR_SHAPE: return "STRATA_ERR_SHAPE";
    case STRATA_ERR_UNSUPPORTED: return "STRATA_ERR_UNSUPPORTED";
    case STRATA_ERR_WORKSPACE: return "STRATA_ERR_WORKSPACE";
    case STRATA_ERR_CUDA: return "STRATA_ERR_CUDA";
    case STRATA_ERR_DEVICE_STATUS: return "STRATA_ERR_DEVICE_STATUS";
    case STRATA_ERR_TIMEOUT: return "STRATA_ERR_TIMEOUT";
    default: return "STRATA_ERR_UNKNOWN";
  }
}

int strata_version(void) { return 100; }

strata_status strata_quantize_groups(const void* w_fp16, int64_t n, int64_t k, int32_t group_size,
                                     uint8_t* codes, void* scales_fp16, uint32_t* dev_status,
                                     strata_stream stream) {
  return strata_quantize_groups_bits(w_fp16, n, k, group_size, 4, codes, scales_fp16, dev_status,
                                     stream);
}

strata_status strata_quantize_groups_bits(const void* w_fp16, int64_t n, int64_t k,
                                          int32_t group_size, int32_t bits, uint8_t* codes,
                                          void* scales_fp16, uint32_t* dev_status,
                                          strata_stream stream) {
  if (group_size != 64 && group_size != 128 && group_size != 256) return STRATA_ERR_UNSUPPORTED;
  if (bits != 4 && bits != 8) return STRATA_ERR_UNSUPPORTED;
  if (n < 0 || k <= 0 || k % group_size) return STRATA_ERR_SHAPE;
  if (n > (int64_t(1) << 40) / k) return STRATA_ERR_SHAPE;
  if (n == 0) return STRATA_OK;
  if (!w_fp16 || !codes || !scales_fp16) return STRATA_ERR_INVALID_ARG;
  if (!aligned(w_fp16, 16) || !aligned(codes, 16) || !aligned(scales_fp16, 2) ||
      (dev_status && !aligned(dev_status, 4)))
    return STRATA_ERR_INVALID_ARG;
  int sms = 0;
  if (device_sms(&sms) != 0) return STRATA_ERR_CUDA;
  return cuda_fail(launch_quantize(w_fp16, n, k, group_size, bits, codes, scales_fp16, dev_status,
                                   reinterpret_cast<cudaStream_t>(stream), sms));
}

size_t strata_route_workspace_size(int64_t T, int32_t E, int32_t k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  // the router scratch depends on H only through the split count; size for the largest split
  return route_layout(T, int64_t(16) * 128, E, k, 0).total;
}

strata_status strata_route_topk(const void* x_bf16, const float* w_router, const float* bias,
                                int64_t T, int64_t H, int32_t E, int32_t k, uint32_t flags,
                                int32_t* ids, float* gates, int32_t* counts, int32_t* offsets,
                                int32_t* perm, int32_t* inv, void* workspace, size_t ws_bytes,
                                strata_stream stream) {
  const strata_status chk = check_route_args(x_bf16, w_router, T, H, E, k, flags, ids, gates,
                                             counts, offsets, perm, inv);
  if (chk != STRATA_OK) return chk;
  const bool all_group = counts && offsets && perm && inv;
  const RouteLayout L = route_layout(T, int64_t(16) * 128, E, k, 0);
  if (!workspace || !aligned(workspace, kAlign)) return STRATA_ERR_WORKSPACE;
  if (ws_bytes < L.total) return STRATA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(base + L.hdr);
  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st) != cudaSuccess) return STRATA_ERR_CUDA;
  if (T == 0) {
    if (all_group) {
      if (cudaMemsetAsync(counts, 0, sizeof(int) * E, st) != cudaSuccess ||
          cudaMemsetAsync(offsets, 0, sizeof(int) * (E + 1), st) != cudaSuccess)
        return STRATA_ERR_CUDA;
    }
    return STRATA_OK;
  }
  int sms = 0;
  if (device_sms(&sms) != 0) return STRATA_ERR_CUDA;
  int nsplit = router_num_splits(T, H, E, sms);
  const int cap = router_num_splits(T, int64_t(16) * 128, E, kRouterSplitsForSizing);
  if (nsplit > cap) nsplit = cap;
  cudaError_t e = launch_router(x_bf16, w_router, bias, T, H, E, k, flags, nsplit,
                                reinterpret_cast<float*>(base + L.partial), ids, gates, st);
  if (e != cudaSuccess) return STRATA_ERR_CUDA;
  if (!all_group) return STRATA_OK;
  PermuteArgs pa{};
  pa.ids = ids;
  pa.T = static_cast<int>(T);
  pa.k = k;
  pa.E = E;
  pa.has_shared = 0;
  pa.counts = counts;
  pa.offsets = offsets;
  pa.perm = perm;
  pa.inv = inv;
  pa.hdr = hdr;
  pa.status = &hdr->status;
  return cuda_fail(launch_permute(pa, st));
}

size_t strata_moe_workspace_size(const strata_moe_layer* layer, int64_t T_max) {
  if (check_layer(layer) != STRATA_OK || T_max < 0 || T_max > kMaxTokens) return 0;
  return fwd_layout(layer, T_max).total;
}

strata_status strata_moe_forward(const strata_moe_layer* layer, const void* x_bf16, int64_t T,
                                 void* out_bf16, void* workspace, size_t ws_bytes,
                                 strata_stream stream) {
  return run_forward(layer, x_bf16, T, out_bf16, nullptr, workspace, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

strata_status strata_moe_forward_padded(const strata_moe_layer* layer, const void* x_bf16,
                                        const int32_t* n_tokens, int64_t T_max, void* out_bf16,
                                        void* workspace, size_t ws_bytes, strata_stream stream) {
  if (!n_tokens || !aligned(n_tokens, 4)) return STRATA_ERR_INVALID_ARG;
  if (T_max < 1) return STRATA_ERR_SHAPE;
  return run_forward(layer, x_bf16, T_max, out_bf16, nullptr, workspace, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream), nullptr, false, nullptr, n_tokens);
}

strata_status strata_moe_forward_ex(const strata_moe_layer* layer, const void* x_bf16, int64_t T,
                                    void* out_bf16, int32_t* ids, float* gates, int32_t* counts,
                                    int32_t* offsets, int32_t* perm, int32_t* inv,
                                    void* workspace, size_t ws_bytes, strata_stream stream) {
  Taps t{ids, gates, counts, offsets, perm, inv};
  return run_forward(layer, x_bf16, T, out_bf16, &t, workspace, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

strata_status strata_moe_forward_stats(const strata_moe_layer* layer, const void* x_bf16,
                                       int64_t T, void* out_bf16, uint64_t* expert_rows,
                                       void* workspace, size_t ws_bytes, strata_stream stream) {
  if (!expert_rows || !aligned(expert_rows, 8)) return STRATA_ERR_INVALID_ARG;
  return run_forward(layer, x_bf16, T, out_bf16, nullptr, workspace, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream), nullptr, false,
                     reinterpret_cast<unsigned long long*>(expert_rows));
}

strata_status strata_moe_forward_profiled(const strata_moe_layer* layer, const void* x_bf16,
                                          int64_t T, void* out_bf16, void* workspace,
                                          size_t ws_bytes, strata_stream stream,
                                          void* const* events, int32_t n_events) {
  if (!events || n_events != STRATA_PROFILE_EVENTS) return STRATA_ERR_INVALID_ARG;
  return run_forward(layer, x_bf16, T, out_bf16, nullptr, workspace, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream), events);
}

size_t strata_moe_stack_workspace_size(const strata_moe_layer* layers, int32_t n_layers,
                                       int64_t T_max) {
  if (!layers || n_layers < 1 || n_layers > 256 || T_max < 0 || T_max > kMaxTokens) return 0;
  size_t ws = 0;
  for (int l = 0; l < n_layers; ++l) {
    if (check_layer(&layers[l]) != STRATA_OK || layers[l].H != layers[0].H) return 0;
    strata_moe_layer L = layers[l];
    L.flags |= STRATA_ADD_RESIDUAL;
    const size_t w = fwd_layout(&L, T_max).total;
    if (w > ws) ws = w;
  }
  return ws + 2 * up(sizeof(uint16_t) * T_max * layers[0].H);  // two activation buffers
}

strata_status strata_moe_stack_forward(const strata_moe_layer* layers, int32_t n_layers,
                                       const void* x_bf16, int64_t T, void* out_bf16,
                                       void* workspace, size_t ws_bytes, strata_stream stream) {
  if (!layers || n_layers < 1 || n_layers > 256) return STRATA_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const strata_status s = check_layer(&layers[l]);
    if (s != STRATA_OK) return s;
    if (layers[l].H != layers[0].H) return STRATA_ERR_SHAPE;
  }
  if (T < 0 || T > kMaxTokens) return STRATA_ERR_SHAPE;
  if (T == 0) return STRATA_OK;
  if (!x_bf16 || !out_bf16 || x_bf16 == out_bf16) return STRATA_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(out_bf16, 16)) return STRATA_ERR_INVALID_ARG;
  const size_t need = strata_moe_stack_workspace_size(layers, n_layers, T);
  if (!workspace || !aligned(workspace, kAlign)) return STRATA_ERR_WORKSPACE;
  if (need == 0 || ws_bytes < need) return STRATA_ERR_WORKSPACE;
  const size_t act = up(sizeof(uint16_t) * T * layers[0].H);
  char* base = static_cast<char*>(workspace);
  const size_t layer_ws = need - 2 * act;
  void* buf[2] = {base + layer_ws, base + layer_ws + act};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const void* cur = x_bf16;
  for (int l = 0; l < n_layers; ++l) {
    strata_moe_layer L = layers[l];
    L.flags |= STRATA_ADD_RESIDUAL;
    void* dst = (l == n_layers - 1) ? out_bf16 : buf[l & 1];
    const strata_status s =
        run_forward(&L, cur, T, dst, nullptr, workspace, layer_ws, st, nullptr, l > 0);
    if (s != STRATA_OK) return s;
    cur = dst;
  }
  return STRATA_OK;
}

size_t strata_moe_host_staging_size(const strata_moe_layer* layer, int64_t T_max) {
  if (check_layer(layer) != STRATA_OK || T_max < 0 || T_max > kMaxTokens) return 0;
  return 2 * up(sizeof(uint16_t) * T_max * layer->H);
}

strata_status strata_moe_forward_host(const strata_moe_layer* layer, const void* x_host,
                                      int64_t T, void* out_host, void* workspace, size_t ws_bytes,
                                      strata_stream stream) {
  strata_status s = check_layer(layer);
  if (s != STRATA_OK) return s;
  if (T < 0 || T > kMaxTokens) return STRATA_ERR_SHAPE;
  if (T == 0) return STRATA_OK;
  if (!x_host || !out_host) return STRATA_ERR_INVALID_ARG;
  const size_t need = strata_moe_workspace_size(layer, T);
  const size_t stage = strata_moe_host_staging_size(layer, T);
  if (!workspace || !aligned(workspace, kAlign)) return STRATA_ERR_WORKSPACE;
  if (ws_bytes < need + stage) return STRATA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(workspace);
  void* xd = base + need;
  void* od = base + need + stage / 2;
  const size_t bytes = sizeof(uint16_t) * T * layer->H;
  if (cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return STRATA_ERR_CUDA;
  s = run_forward(layer, xd, T, od, nullptr, workspace, need, st);
  if (s != STRATA_OK) return s;
  if (cudaMemcpyAsync(out_host, od, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return STRATA_ERR_CUDA;
  return cuda_fail(cudaStreamSynchronize(st));
}

strata_status strata_read_status(uint32_t* dev_status, strata_stream stream, uint32_t* status_out) {
  if (!dev_status || !status_out) return STRATA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return STRATA_ERR_CUDA;
  if (cudaMemsetAsync(dev_status, 0, sizeof(uint32_t), st) != cudaSuccess) return STRATA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return STRATA_ERR_CUDA;
  *status_out = v;
  if (v == 0) return STRATA_OK;
  return (v & STRATA_DEV_TIMEOUT) ? STRATA_ERR_TIMEOUT : STRATA_ERR_DEVICE_STATUS;
}

strata_status strata_group_rows(const int32_t* ids, int64_t T, int32_t k, int32_t E,
                                int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                void* workspace, size_t ws_bytes, strata_stream stream) {
  if (T < 0 || T > kMaxTokens) return STRATA_ERR_SHAPE;
  if (k < 1 || k > STRATA_MAX_TOPK || E < 1 || E > STRATA_MAX_EXPERTS) return STRATA_ERR_INVALID_ARG;
  if (!counts || !offsets || (T > 0 && (!ids || !perm || !inv))) return STRATA_ERR_INVALID_ARG;
  if ((ids && !aligned(ids, 4)) || !aligned(counts, 4) || !aligned(offsets, 4) ||
      (perm && !aligned(perm, 4)) || (inv && !aligned(inv, 4)))
    return STRATA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, kAlign) || ws_bytes < STRATA_GROUP_WORKSPACE_BYTES)
    return STRATA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st) != cudaSuccess) return STRATA_ERR_CUDA;
  PermuteArgs pa{};
  pa.ids = ids;
  pa.T = static_cast<int>(T);
  pa.k = k;
  pa.E = E;
  pa.counts = counts;
  pa.offsets = offsets;
  pa.perm = perm;
  pa.inv = inv;
  pa.hdr = hdr;
  pa.status = &hdr->status;
  return cuda_fail(launch_permute(pa, st));
}

strata_status strata_selftest_bounded_waits(uint32_t* dev_words, int64_t limit_cycles,
                                            strata_stream stream) {
  if (!dev_words || !aligned(dev_words, 16)) return STRATA_ERR_INVALID_ARG;
  if (limit_cycles < 1 || limit_cycles > tc::kWaitCycles) return STRATA_ERR_INVALID_ARG;
  return cuda_fail(launch_wait_selftest(dev_words, limit_cycles,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

strata_status strata_workspace_status(void* workspace, strata_stream stream, uint32_t* status_out) {
  if (!workspace || !aligned(workspace, kAlign)) return STRATA_ERR_WORKSPACE;
  return strata_read_status(&reinterpret_cast<WsHeader*>(workspace)->status, stream, status_out);
}

}  // extern "C"
