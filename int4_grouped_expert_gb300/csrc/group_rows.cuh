// Stable counting sort of the routed rows by expert, shared by the stand-alone grouping kernel and
// the last CTA of the fused decode router. Tokens routed to the same expert become one contiguous
// segment of the grouped GEMM ("Strata" 3090 tuning, xdnf.cn/news/329730, §3.2).
//
// Rows r = t*k + j of the flattened [T, k] id array are ordered by (expert, token): each warp owns a
// contiguous range of r, counts it into its own histogram row (equal ids inside a 32-row step are
// grouped with __match_any_sync), the histograms are scanned per expert in warp order, and the same
// walk then hands out positions. The result does not depend on thread timing. Everything the CTA
// reads back lives in shared memory; global memory only receives the outputs.
#pragma once

#include "kernels.cuh"

namespace strata {

// Exclusive scan of one int per thread over the whole block (blockDim.x = 32 * NW);
// scratch holds NW + 1 ints. Every thread of the block must call it.
template <int NW>
__device__ __forceinline__ int block_scan_excl(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < NW ? scratch[lane] : 0;
    int winc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += n;
    }
    if (lane < NW) scratch[lane] = winc - w;
    if (lane == 31) scratch[NW] = winc;
  }
  __syncthreads();
  const int res = scratch[warp] + inc - v;
  *total = scratch[NW];
  __syncthreads();
  return res;
}

// Shared-memory scratch of group_rows (ints).
struct GroupSmem {
  int* hist;    // [NW][E]
  int* cnt;     // [E]
  int* off;     // [E + 1]
  int* seg_e;   // [E + 2]
  int* seg_r0;  // [E + 2]
  int* seg_n;   // [E + 2]
  int* scratch; // [NW + 1]
};
__host__ __device__ constexpr size_t group_smem_ints(int NW, int E) {
  return static_cast<size_t>(NW) * E + E + (E + 1) + 3 * (E + 2) + NW + 1;
}
__device__ __forceinline__ GroupSmem carve_group_smem(int* base, int NW, int E) {
  GroupSmem g;
  g.hist = base;
  g.cnt = g.hist + NW * E;
  g.off = g.cnt + E;
  g.seg_e = g.off + E + 1;
  g.seg_r0 = g.seg_e + E + 2;
  g.seg_n = g.seg_r0 + E + 2;
  g.scratch = g.seg_n + E + 2;
  return g;
}

// ids: the [T, k] ids (global or shared memory).
// The split-K arrival counters of nchunks chunks, zeroed by threads tid = 0 .. nt - 1 (16-byte
// stores when the count and the base allow them).
__device__ __forceinline__ void zero_split_counters(const PermuteArgs& a, int nchunks, int tid,
                                                    int nt) {
  const int n = nchunks * a.cnt_per_chunk;
  if ((n & 3) == 0 && (reinterpret_cast<uintptr_t>(a.split_cnt) & 15) == 0) {
#pragma unroll 1
    for (int i = tid; i < n / 4; i += nt) reinterpret_cast<int4*>(a.split_cnt)[i] = make_int4(0, 0, 0, 0);
  } else {
#pragma unroll 1
    for (int i = tid; i < n; i += nt) a.split_cnt[i] = 0;
  }
}

template <int NW>
__device__ void group_rows(const PermuteArgs& a, const int* ids, GroupSmem sm) {
  constexpr int NT = NW * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E;
  const int R = a.T * a.k;
  int* hist = sm.hist;
  for (int i = tid; i < NW * E; i += NT) hist[i] = 0;
  __syncthreads();

  const int per_warp = (R + NW - 1) / NW;
  const int rbeg = min(R, warp * per_warp), rend = min(R, rbeg + per_warp);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = rbeg; base < rend; base += 32) {
    const int r = base + lane;
    const unsigned active = __ballot_sync(0xffffffffu, r < rend);
    if (r < rend) {
      int e = ids[r];
      if (e < 0 || e >= E) {
        set_status(a.status, STRATA_DEV_BAD_ID);
        e = -1;
      }
      const unsigned m = __match_any_sync(active, e);
      if (e >= 0 && (m & lt_mask) == 0) hist[warp * E + e] += __popc(m);
      __syncwarp(active);
    }
  }
  __syncthreads();

  const int ept = (E + NT - 1) / NT;
  const int e0 = min(E, tid * ept), e1 = min(E, e0 + ept);
  int my = 0;
  for (int e = e0; e < e1; ++e)
    for (int w = 0; w < NW; ++w) my += hist[w * E + e];
  int total;
  int run = block_scan_excl<NW>(my, sm.scratch, &total);
  for (int e = e0; e < e1; ++e) {
    int c = 0;
    for (int w = 0; w < NW; ++w) {
      const int h = hist[w * E + e];
      hist[w * E + e] = run + c;
      c += h;
    }
    sm.cnt[e] = c;
    sm.off[e] = run;
    a.counts[e] = c;
    a.offsets[e] = run;
    if (a.hits && c > 0) atomicAdd(a.hits + e, static_cast<unsigned long long>(c));
    run += c;
  }
  if (a.hits && a.has_shared && tid == 0 && a.T > 0)
    atomicAdd(a.hits + E, static_cast<unsigned long long>(a.T));
  if (tid == 0) {
    a.offsets[E] = total;
    sm.off[E] = total;
  }
  __syncthreads();

  for (int base = rbeg; base < rend; base += 32) {
    const int r = base + lane;
    const unsigned active = __ballot_sync(0xffffffffu, r < rend);
    if (r < rend) {
      int e = ids[r];
      if (e < 0 || e >= E) e = -1;
      const unsigned m = __match_any_sync(active, e);
      if (e >= 0) {
        const int pos = hist[warp * E + e] + __popc(m & lt_mask);
        a.perm[pos] = r / a.k;
        a.inv[r] = pos;
      } else {
        a.inv[r] = -1;  // left out of every group
      }
      __syncwarp(active);
      if (e >= 0 && (m & lt_mask) == 0) hist[warp * E + e] += __popc(m);
      __syncwarp(active);
    }
  }
  if (a.has_shared)
    for (int t = tid; t < a.T; t += NT) a.perm[R + t] = t;
  __syncthreads();

  if (a.seg_expert == nullptr) return;
  // Active segments: the shared expert first (the largest), then routed experts with rows, by id.
  const int sh = (a.has_shared && a.T > 0) ? 1 : 0;
  int nz = 0;
  for (int e = e0; e < e1; ++e) nz += (sm.cnt[e] > 0);
  int nseg_routed;
  int sidx = block_scan_excl<NW>(nz, sm.scratch, &nseg_routed) + sh;
  for (int e = e0; e < e1; ++e) {
    const int c = sm.cnt[e];
    if (c > 0) {
      sm.seg_e[sidx] = e;
      sm.seg_r0[sidx] = sm.off[e];
      sm.seg_n[sidx] = c;
      ++sidx;
    }
  }
  const int nseg = nseg_routed + sh;
  if (sh && tid == 0) {
    sm.seg_e[0] = E;
    sm.seg_r0[0] = R;
    sm.seg_n[0] = a.T;
  }
  __syncthreads();
  for (int s = tid; s < nseg; s += NT) {
    a.seg_expert[s] = sm.seg_e[s];
    a.seg_row0[s] = sm.seg_r0[s];
    a.seg_rows[s] = sm.seg_n[s];
  }
  const int spt = (nseg + NT - 1) / NT;
  const int s0 = min(nseg, tid * spt), s1 = min(nseg, s0 + spt);
  if (a.chunk_list) {
    // Warp path: a flat list of tokc-row chunks; items = chunk x row tile (x contraction split).
    int my_c = 0;
    for (int s = s0; s < s1; ++s) my_c += (sm.seg_n[s] + a.tokc - 1) / a.tokc;
    int nchunks;
    int off = block_scan_excl<NW>(my_c, sm.scratch, &nchunks);
    for (int s = s0; s < s1; ++s) {
      const int e = sm.seg_e[s], row0 = sm.seg_r0[s], rows = sm.seg_n[s];
      for (int c = 0; c * a.tokc < rows; ++c)
        a.chunk_list[off++] = make_int4(e, row0 + c * a.tokc, min(a.tokc, rows - c * a.tokc), 0);
    }
    if (tid == 0) {
      a.hdr->nseg = nseg;
      a.hdr->n_chunks = nchunks;
      a.hdr->n_items_gu = nchunks * a.mtiles_gu * a.ksplit_gu;
      a.hdr->n_items_dn = nchunks * a.mtiles_dn * a.ksplit_dn;
      a.hdr->next_gu = 0;
      a.hdr->next_dn = 0;
    }
    if (a.split_cnt) zero_split_counters(a, nchunks, tid, NT);
    return;
  }
  // Tensor-core path: tiles per segment = (token chunks) x (row tiles); prefix over segments.
  int my_gu = 0, my_dn = 0;
  for (int s = s0; s < s1; ++s) {
    const int chunks = (sm.seg_n[s] + a.tokc - 1) / a.tokc;
    my_gu += chunks * a.mtiles_gu;
    my_dn += chunks * a.mtiles_dn;
  }
  int tot_gu, tot_dn;
  int pg = block_scan_excl<NW>(my_gu, sm.scratch, &tot_gu);
  int pd = block_scan_excl<NW>(my_dn, sm.scratch, &tot_dn);
  for (int s = s0; s < s1; ++s) {
    const int chunks = (sm.seg_n[s] + a.tokc - 1) / a.tokc;
    a.seg_item_gu[s] = pg;
    a.seg_item_dn[s] = pd;
    pg += chunks * a.mtiles_gu;
    pd += chunks * a.mtiles_dn;
  }
  if (tid == 0) {
    a.seg_item_gu[nseg] = tot_gu;
    a.seg_item_dn[nseg] = tot_dn;
    a.hdr->nseg = nseg;
    a.hdr->n_items_gu = tot_gu;
    a.hdr->n_items_dn = tot_dn;
    a.hdr->next_gu = 0;
    a.hdr->next_dn = 0;
  }
}

// ----------------------------------------------------------------------------- small batches
// The same grouping for the warp path when the routed rows are few (R = T*k <= 512), written for
// the one CTA that runs it once per layer: every loop is rolled, so the code the CTA fetches stays
// small. Rows are marked in a per-expert bitmask (atomicOr: order-free), a row's position is the
// expert's offset plus the marked rows below it, and one scan over the experts yields offsets,
// segment indices and chunk offsets together. Outputs are identical to group_rows.
constexpr int kGroupSmallMaxR = 512;
__host__ __device__ constexpr size_t group_small_ints(int NW, int E, int R) {
  return static_cast<size_t>(E) * ((R + 31) / 32) + (E + 1) + 2 * (NW + 1) + 1;
}

// Exclusive block scan of a 64-bit value (blockDim.x = 32 * NW); scratch holds 2 * (NW + 1) ints.
template <int NW>
__device__ __forceinline__ unsigned long long block_scan_excl64(unsigned long long v, int* scratch,
                                                                unsigned long long* total) {
  unsigned long long* sc = reinterpret_cast<unsigned long long*>(scratch);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) sc[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = lane < NW ? sc[lane] : 0ull;
    unsigned long long winc = w;
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long n = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += n;
    }
    __syncwarp();
    if (lane < NW) sc[lane] = winc - w;
    if (lane == 31) sc[NW] = winc;
  }
  __syncthreads();
  const unsigned long long res = sc[warp] + inc - v;
  *total = sc[NW];
  return res;
}

// ids: the [T, k] ids in shared memory; smem: group_small_ints(NW, E, T*k) ints, 8-byte aligned.
template <int NW>
__device__ void group_rows_small(const PermuteArgs& a, const int* ids, int* smem) {
  constexpr int NT = NW * 32;
  const int tid = threadIdx.x;
  const int E = a.E, R = a.T * a.k, MW = (R + 31) / 32;
  uint32_t* mask = reinterpret_cast<uint32_t*>(smem);  // [E][MW]
  int* off = smem + E * MW;                              // [E + 1]
  int* scratch = off + E + 1;
  scratch += (reinterpret_cast<uintptr_t>(scratch) & 7) ? 1 : 0;
#pragma unroll 1
  for (int i = tid; i < E * MW; i += NT) mask[i] = 0u;
  __syncthreads();
#pragma unroll 1
  for (int r = tid; r < R; r += NT) {
    const int e = ids[r];
    if (e < 0 || e >= E) set_status(a.status, STRATA_DEV_BAD_ID);
    else atomicOr(&mask[e * MW + (r >> 5)], 1u << (r & 31));
  }
  __syncthreads();
  // experts [e0, e1) of this thread: rows, active segments, chunks, packed 21 bits apart
  const int ept = (E + NT - 1) / NT;
  const int e0 = min(E, tid * ept), e1 = min(E, e0 + ept);
  unsigned long long mine = 0ull;
#pragma unroll 1
  for (int e = e0; e < e1; ++e) {
    int c = 0;
#pragma unroll 1
    for (int w = 0; w < MW; ++w) c += __popc(mask[e * MW + w]);
    if (c > 0) mine += static_cast<unsigned long long>(c) |
                       (1ull << 21) | (static_cast<unsigned long long>((c + a.tokc - 1) / a.tokc) << 42);
  }
  unsigned long long tot;
  unsigned long long run = block_scan_excl64<NW>(mine, scratch, &tot);
  const int sh = (a.has_shared && a.T > 0) ? 1 : 0;
  const int sh_chunks = sh ? (a.T + a.tokc - 1) / a.tokc : 0;
  const int nseg = static_cast<int>((tot >> 21) & 0x1FFFFF) + sh;
  const int nchunks = static_cast<int>(tot >> 42) + sh_chunks;
#pragma unroll 1
  for (int e = e0; e < e1; ++e) {
    int c = 0;
#pragma unroll 1
    for (int w = 0; w < MW; ++w) c += __popc(mask[e * MW + w]);
    const int row0 = static_cast<int>(run & 0x1FFFFF);
    off[e] = row0;
    a.counts[e] = c;
    a.offsets[e] = row0;
    if (a.hits && c > 0) atomicAdd(a.hits + e, static_cast<unsigned long long>(c));
    if (c > 0) {
      const int sidx = static_cast<int>((run >> 21) & 0x1FFFFF) + sh;
      a.seg_expert[sidx] = e;
      a.seg_row0[sidx] = row0;
      a.seg_rows[sidx] = c;
      int ch = static_cast<int>(run >> 42) + sh_chunks;
#pragma unroll 1
      for (int q = 0; q * a.tokc < c; ++q)
        a.chunk_list[ch++] = make_int4(e, row0 + q * a.tokc, min(a.tokc, c - q * a.tokc), 0);
      run += static_cast<unsigned long long>(c) | (1ull << 21) |
             (static_cast<unsigned long long>((c + a.tokc - 1) / a.tokc) << 42);
    }
  }
  if (tid == 0) {
    if (a.hits && sh) atomicAdd(a.hits + E, static_cast<unsigned long long>(a.T));
    a.offsets[E] = static_cast<int>(tot & 0x1FFFFF);
    if (sh) {
      a.seg_expert[0] = E;
      a.seg_row0[0] = R;
      a.seg_rows[0] = a.T;
    }
    a.hdr->nseg = nseg;
    a.hdr->n_chunks = nchunks;
    a.hdr->n_items_gu = nchunks * a.mtiles_gu * a.ksplit_gu;
    a.hdr->n_items_dn = nchunks * a.mtiles_dn * a.ksplit_dn;
    a.hdr->next_gu = 0;
    a.hdr->next_dn = 0;
  }
#pragma unroll 1
  for (int q = tid; q < sh_chunks; q += NT)
    a.chunk_list[q] = make_int4(E, R + q * a.tokc, min(a.tokc, a.T - q * a.tokc), 0);
  if (a.split_cnt) zero_split_counters(a, nchunks, tid, NT);
  __syncthreads();
  // positions: expert offset + marked rows of that expert below r (stable by token)
#pragma unroll 1
  for (int r = tid; r < R; r += NT) {
    const int e = ids[r];
    if (e < 0 || e >= E) {
      a.inv[r] = -1;  // left out of every group
      continue;
    }
    const uint32_t* m = mask + e * MW;
    int pos = off[e] + __popc(m[r >> 5] & ((1u << (r & 31)) - 1u));
#pragma unroll 1
    for (int w = 0; w < (r >> 5); ++w) pos += __popc(m[w]);
    a.perm[pos] = r / a.k;
    a.inv[r] = pos;
  }
  if (a.has_shared) {
#pragma unroll 1
    for (int t = tid; t < a.T; t += NT) a.perm[R + t] = t;
  }
}

}  // namespace strata
