// Launchers and argument blocks shared between the kernels and the C ABI layer.
#pragma once

#include "common.cuh"

namespace strata {

struct PermuteArgs {
  const int* ids;
  int T, k, E, has_shared;
  int* counts;   // [E]
  int* offsets;  // [E+1]
  int* perm;     // [T*k + T]: rows of the shared segment follow the routed rows
  int* inv;      // [T*k]
  // grouped-GEMM work lists (optional: seg_expert == nullptr skips them)
  int* seg_expert;
  int* seg_row0;
  int* seg_rows;
  int* seg_item_gu;  // [nseg + 1] exclusive prefix of gate/up items
  int* seg_item_dn;  // [nseg + 1]
  int tokc;          // rows per work item along the token dimension
  int mtiles_gu;     // gate/up row tiles per expert
  int mtiles_dn;     // down row tiles per expert
  int ksplit_gu;     // gate/up contraction splits per tile (1 = none)
  int ksplit_dn;     // down contraction splits per tile (1 = none)
  int cnt_per_chunk; // split-K arrival counters per chunk (zeroed here)
  int* split_cnt;    // arrival counters of the split-K reductions
  unsigned long long* hits;  // optional [E + has_shared]: += rows routed to each expert (statistics)
  int4* chunk_list;  // warp path: {expert, first row, rows, 0} per tokc-row chunk (else null)
  WsHeader* hdr;
  uint32_t* status;
};

struct GemmArgs {
  const uint8_t* codes0;     // gate (gate/up mode) or down codes, [experts, N, K/2]
  const __half* scales0;     // [experts, N, K/128]
  const uint8_t* codes1;     // up codes (gate/up mode)
  const __half* scales1;
  const __nv_bfloat16* act;  // gate/up: x [T, K]; down: h [rows, K]; pair-interleaved chunks,
                             // f16 for the CTA-staged kernel (the type only sets the stride)
  const int* perm;           // token (activation row) of each GEMM row, or null: row = activation row
  void* out;                 // gate/up: h [rows, N] (f16 from the CTA-staged kernel, bf16 from the
                             // per-warp one); down: y fp32 [rows, N]
  int K;                     // contraction length (H for gate/up, I for down)
  int N;                     // weight rows per expert (I for gate/up, H for down)
  WsHeader* hdr;
  const int* seg_expert;
  const int* seg_row0;
  const int* seg_rows;
  const int* seg_item;       // exclusive prefix of work items per segment, [nseg + 1]
  const int4* chunk_list;    // {expert, first row, rows, 0} per 8-row chunk
  int ksplit;                // contraction splits per tile (gate/up only)
  // f16 operands (CTA-staged kernel): activation row r (perm[r] when perm is set) is stored as
  // act * 2^-aexp[.] and the result is multiplied back; gate/up stores h row r as h * 2^-2a and
  // writes 2a to hexp[r] (each may be null: exponent 0)
  const int* aexp;
  int* hexp;
  int group;                 // scale group size: 64, 128 or 256 (CTA-staged kernel; others 128)
  float* split_part;         // [tiles * ksplit * 256] partial sums of split tiles
  int* split_cnt;            // [tiles] arrival counters (zero on entry)
};

// Tensor-core grouped GEMM (gemm_tc.cu).
struct TcArgs {
  const uint8_t* codes0;  // gate or down codes [experts, Nw, K/2]
  const __half* scales0;
  const uint8_t* codes1;  // up codes (gate/up)
  const __half* scales1;
  void* out;              // gate/up: h f16 [rows, Nw] (pair-interleaved columns); down: y fp32
  int K, Nw;              // contraction; weight rows per expert
  int group;              // scale group size: 64, 128 or 256
  int bits;               // code width: 4 (codes [.., K/2]) or 8 (codes [.., K])
  const int* aexp;        // range exponent of each B row (null: 0), as GemmArgs::aexp
  int* hexp;              // gate/up: 2a of each h row (null: not written)
  WsHeader* hdr;
  const int* seg_expert;
  const int* seg_row0;
  const int* seg_rows;
  const int* seg_item;    // exclusive prefix of tiles per segment
  uint32_t* status;
};

// Fused decode router: logits (split along H over the grid), then the last CTA does softmax +
// top-k for every token and groups the rows.
struct RouteSmallArgs {
  const __nv_bfloat16* x;  // [T, H]
  const void* wr;          // [E, H] fp32, or fp16 with wr_fp16
  bool wr_fp16;
  const float* bias;       // [E] or null
  int T, H, E, k;          // T: tokens, or the maximum when T_dev is set
  const int* T_dev;        // optional device token count (live rows 0..*T_dev-1 of x), or null
  uint32_t flags;
  int epc;                 // experts per CTA (each split over 8 / epc warps along H)
  void* x_perm;            // [T, H]: x with every 8-wide chunk in (0,4,1,5,2,6,3,7) order, or null
  bool x_f16;              // x_perm as f16 (CTA-staged GEMM) instead of bf16 (per-warp GEMM)
  int* xexp;               // x_f16: [T] range exponent of each token's row of x_perm (range_exp)
  float* logits;           // [T][E] scratch
  int* ids;
  float* gates;
  PermuteArgs grp;         // grouping of the rows (ids = this->ids)
  bool do_group;
};

cudaError_t launch_quantize(const void* w, int64_t n, int64_t k, int group, int bits,
                            uint8_t* codes, void* scales, uint32_t* status, cudaStream_t stream,
                            int num_sms);
int router_num_splits(int64_t T, int64_t H, int E, int num_sms);
cudaError_t launch_router(const void* x, const void* wr, const float* bias, int64_t T, int64_t H,
                          int E, int k, uint32_t flags, int nsplit, float* partial, int* ids,
                          float* gates, cudaStream_t stream);
cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t stream);
constexpr int kRouteSmallMaxT = 64;  // tokens handled by the fused decode router
int route_small_epc(int E, int num_sms);
cudaError_t launch_route_small(const RouteSmallArgs& a, cudaStream_t stream);
cudaError_t launch_gemm_warp(const GemmArgs& a, bool gate_up, int num_sms, cudaStream_t stream);
// CTA-staged warp GEMM (gemm_cta.cu): row blocks of cta_gemm_block_rows() weight rows per item.
int cta_gemm_block_rows(bool gate_up);
int cta_gemm_warps();
int cta_gemm_ksplit(int64_t items, int64_t K, int num_sms);
// even: the equal-stage-range schedule (cta_gemm_even), which needs cta_gemm_partial_floats(num_sms)
// floats of split_part and one split_cnt counter per (chunk, row block, consumer warp)
bool cta_gemm_even(int64_t max_tiles, int num_sms);
int64_t cta_gemm_partial_floats(int num_sms);
cudaError_t launch_gemm_cta(const GemmArgs& a, bool gate_up, int64_t experts, int num_sms,
                            bool even, cudaStream_t stream);
int warp_ksplit(int64_t T, int E, int k, int shared, int64_t I, int64_t H);
constexpr int kTcRows = 256;      // token rows per tensor-core tile
constexpr int kTcRowsSmall = 64;  // the same for batches with few rows per expert
// b_rows: the B operand rows [rows, K] bf16; experts: weight matrices per code tensor
// (routed + shared); tile_rows: kTcRows or kTcRowsSmall (the grouping's chunk size)
cudaError_t launch_gemm_tc(const TcArgs& a, bool gate_up, const void* b_rows, int64_t rows,
                           int64_t experts, int tile_rows, int num_sms, cudaStream_t stream);
// xp[r] = x[perm[r]], each 8-wide chunk in the order (and type) its GEMM reads: mode 0 bf16 for
// the per-warp decode GEMM, 1 f16 for the CTA-staged decode GEMM, 2 f16 for the tensor-core GEMM
constexpr int kGatherWarp = 0, kGatherCta = 1, kGatherTc = 2;
// rexp: f16 modes, the range exponent of each gathered row (see range_exp), or null
cudaError_t launch_gather_rows(const void* x, const int* perm, int64_t rows, int64_t H, void* xp,
                               int mode, int* rexp, cudaStream_t stream);
// Argument checks shared by the router entry points (strata_api.cu).
strata_status check_route_args(const void* x_bf16, const void* w_router, int64_t T, int64_t H,
                               int32_t E, int32_t k, uint32_t flags, const int32_t* ids,
                               const float* gates, const int32_t* counts, const int32_t* offsets,
                               const int32_t* perm, const int32_t* inv);
// T_dev (optional): the live token count on the device; T is then the maximum, R is taken as
// live * k and rows of out beyond the live tokens are left untouched
// selftest.cu: both bounded waits on things nothing completes (see strata_selftest_bounded_waits)
cudaError_t launch_wait_selftest(uint32_t* words, long long limit, cudaStream_t stream);
cudaError_t launch_combine(const float* y, const float* gates, const int* inv, const void* x,
                           int64_t T, int64_t H, int k, int has_shared, int64_t R, int residual,
                           void* out, const int* T_dev, cudaStream_t stream);

}  // namespace strata
