/*
 * strata.h — C ABI of the GB300 routed MoE FFN layer with int4 group-quantized experts.
 *
 * The operations follow the problem statement of five write-ups about the
 * "Strata" MoE engine (the pages have no titles; each is named by its address):
 *   [tuning-3090] xdnf.cn/news/329730            §3.2 tokens routed to one expert are
 *                                                gathered into one group of a single
 *                                                grouped-GEMM launch; §5.2 fixed,
 *                                                pre-allocated buffers
 *   [tuning-moe]  lpnh.cn/news/2730718           §2.1 group_quantize(weight, 128, 4):
 *                                                scale = absmax/7, clamp(-8, 7);
 *                                                §2.3 point 1: router softmax + top-k
 *                                                fused in one kernel
 *   [tok-102]     zwxr.cn/news/276292            §3.2 routing engine: logits in,
 *                                                softmax, partial sort, expert ids out
 *   [glm-4090]    haowenji.com/articles/x-2109226022155796480
 *                                                §01 experts are Gate/Up + Down
 *                                                projections; 8 routed + 1 shared
 *                                                expert per token
 *
 * Conventions for every call below.
 *  - All tensor pointers are DEVICE pointers owned by the caller, unless a
 *    parameter says "host". The library never allocates or frees memory and keeps
 *    no state between calls; scratch memory is a caller-owned workspace whose size
 *    the *_workspace_size queries return.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) unless documented as blocking.
 *  - Arguments are validated on the host before anything is launched; a failed
 *    check returns its status and has no side effects.
 *  - Launch failures return STRATA_ERR_CUDA (from cudaGetLastError).
 *  - Kernels never trap. Faults they detect in the data (a non-finite weight, an
 *    expert id out of range) set bits in a device status word, read back with
 *    strata_workspace_status / strata_read_status (these synchronize the stream).
 *  - Dtypes: bf16/fp16 tensors are passed as void* to raw 16-bit storage.
 *  - Layouts are row-major and contiguous unless stated.
 */
#ifndef STRATA_H_
#define STRATA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* strata_stream; /* identical to cudaStream_t */

typedef enum {
  STRATA_OK = 0,
  STRATA_ERR_INVALID_ARG = 1,   /* null pointer, bad flag, k > E, ... */
  STRATA_ERR_SHAPE = 2,         /* a dimension is not a multiple of 128, or out of range */
  STRATA_ERR_UNSUPPORTED = 3,   /* group size not 64/128/256, or a size above a limit */
  STRATA_ERR_WORKSPACE = 4,     /* workspace null, misaligned or smaller than required */
  STRATA_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
  STRATA_ERR_DEVICE_STATUS = 6, /* the device status word reported a data fault */
  STRATA_ERR_TIMEOUT = 7        /* a bounded device-side wait gave up */
} strata_status;

/* Flags of strata_route_topk / strata_moe_layer.flags. */
#define STRATA_RENORM 0x1u       /* renormalise the k gates of a token to sum to 1 (off by default:
                                    the pages never renormalise) */
#define STRATA_ADD_RESIDUAL 0x2u /* moe_forward only: out = bf16(x + MoE(x)), one rounding */
#define STRATA_ROUTER_FP16 0x4u  /* the router weights are fp16 [E, H] instead of fp32 ("Strata" MoE
                                    tuning notes, lpnh.cn/news/2730718, §2.1: the router kept in
                                    fp16); logits still accumulate in fp32 over exact products */
/* Kernel-path selection of moe_forward (results agree within the layer tolerance; default: the
   tensor-core path from 128 tokens up, the warp path below). For tests and tuning. */
#define STRATA_FORCE_WARP_PATH 0x100u /* mma.sync warp GEMMs, B from registers */
#define STRATA_FORCE_TC_PATH 0x200u   /* tcgen05 / TMEM GEMMs fed by TMA */
/* Forward entry points: the caller promises that the workspace is zero-filled or was last used by
   a completed forward call (of any layer) that reported no device timeout. The per-call clearing
   of the workspace header (one memset between the previous kernel and the router) is then
   skipped; the device status word is not cleared per call either, but accumulates until
   strata_workspace_status reads (and clears) it. After a call that timed out, zero the workspace
   again before reusing it with this flag. */
#define STRATA_WS_REUSE 0x8u

/* Bits of the device status word. */
#define STRATA_DEV_NONFINITE 0x1u /* a quantized group held inf/nan (its scale is written as NaN,
                                     its codes as 0) */
#define STRATA_DEV_BAD_ID 0x2u    /* an expert id outside [0, E) reached the permutation */
#define STRATA_DEV_TIMEOUT 0x4u   /* a bounded device wait gave up */
#define STRATA_DEV_BAD_TOKENS 0x8u /* strata_moe_forward_padded: the device token count was outside
                                      [0, T_max]; the call ran with no live token */

#define STRATA_GROUP 128     /* [tuning-moe] §2.1: 128 weights share one scale */
#define STRATA_MAX_EXPERTS 1024
#define STRATA_MAX_TOPK 32

/* Human-readable name of a status code (static string, never NULL). */
const char* strata_status_string(int status);

/* ABI version: major*10000 + minor*100 + patch. */
int strata_version(void);

/*
 * strata_quantize_groups — symmetric int4 group quantization, [tuning-moe] §2.1.
 *
 * For each row i of w and each group g of G = group_size consecutive columns:
 *   scale[i,g] = fp16_round_nearest_even(absmax(w[i, Gg : Gg+G]) / 7)
 *   q[i,c]     = clamp(round_half_even(w[i,c] / scale[i,g]), -8, 7)   (exact quotient)
 *   a group whose stored scale is 0 gets q = 0.
 * w_fp16      [n, k] fp16, row-major (device).
 * codes       [n, k/2] uint8 (device, written): byte c of row i holds q[i,2c] in bits 0-3 and
 *             q[i,2c+1] in bits 4-7, as 4-bit two's complement.
 * scales_fp16 [n, k/group_size] fp16 (device, written).
 * group_size  128 (the pages' choice) or 64 / 256 (the sizes they weigh against it);
 *             anything else -> STRATA_ERR_UNSUPPORTED; k % group_size != 0 -> STRATA_ERR_SHAPE;
 *             n == 0 is a no-op.
 * dev_status  optional device uint32 (NULL to skip): STRATA_DEV_NONFINITE is OR-ed in when a
 *             group holds inf/nan; such a group gets scale NaN and codes 0.
 * Buffers must be 16-byte aligned (STRATA_ERR_INVALID_ARG otherwise).
 */
strata_status strata_quantize_groups(const void* w_fp16, int64_t n, int64_t k, int32_t group_size,
                                     uint8_t* codes, void* scales_fp16, uint32_t* dev_status,
                                     strata_stream stream);

/*
 * strata_quantize_groups_bits — the same with the sketch's bit width as a parameter
 * ([tuning-moe] §2.1: scale = absmax / (2^(bits-1) - 1); the pages keep experts at 4 bits and
 * attention projections at 8).
 * bits  4: exactly strata_quantize_groups.
 *       8: scale[i,g] = fp16_round_nearest_even(absmax / 127),
 *          q[i,c] = clamp(round_half_even(w[i,c] / scale[i,g]), -128, 127) (exact quotient);
 *          codes [n, k] int8 (two's complement), one per byte, row-major.
 *       anything else -> STRATA_ERR_UNSUPPORTED.
 * Other arguments, errors and alignment as strata_quantize_groups.
 */
strata_status strata_quantize_groups_bits(const void* w_fp16, int64_t n, int64_t k,
                                          int32_t group_size, int32_t bits, uint8_t* codes,
                                          void* scales_fp16, uint32_t* dev_status,
                                          strata_stream stream);

/*
 * strata_route_topk — router GEMV + softmax + top-k + token grouping,
 * [tuning-moe] §2.3 point 1 and [tok-102] §3.2; grouping per [tuning-3090] §3.2.
 *
 *   logits[t,e] = sum_h x[t,h] * w_router[e,h] + bias[e]     (fp32 accumulation)
 *   p[t,:]      = softmax(logits[t,:])                        (fp32)
 *   ids[t,:]    = the k experts of largest logit, in descending order, ties to the lower id
 *   gates[t,j]  = p[t, ids[t,j]]   (divided by sum_j of them when flags & STRATA_RENORM)
 * and, when the pointers are non-NULL, the grouping of the T*k routed rows by expert, rows
 * ordered by (expert, token):
 *   counts[e]   rows routed to expert e;  offsets[e] = sum_{e'<e} counts[e'], offsets[E] = T*k
 *   perm[r]     token of row r;           inv[t,j] = row of (t, ids[t,j])
 * x_bf16 [T,H] bf16; w_router [E,H] fp32 (fp16 when flags & STRATA_ROUTER_FP16: cast the
 * pointer); bias [E] fp32 or NULL. flags: STRATA_RENORM | STRATA_ROUTER_FP16.
 * ids [T,k] int32, gates [T,k] fp32 (required); counts [E], offsets [E+1], perm [T*k],
 * inv [T,k] int32 (optional as a group: all four or none).
 * Limits: H % 128 == 0, 1 <= k <= min(E, 32), E <= 1024, T >= 0 (T == 0 writes counts/offsets
 * as zeros only). workspace >= strata_route_workspace_size(T, E, k) bytes, 256-byte aligned.
 */
size_t strata_route_workspace_size(int64_t T, int32_t E, int32_t k);
strata_status strata_route_topk(const void* x_bf16, const float* w_router, const float* bias,
                                int64_t T, int64_t H, int32_t E, int32_t k, uint32_t flags,
                                int32_t* ids, float* gates, int32_t* counts, int32_t* offsets,
                                int32_t* perm, int32_t* inv, void* workspace, size_t ws_bytes,
                                strata_stream stream);

/*
 * strata_route_topk_noalloc — strata_route_topk without a workspace argument, for callers that
 * may not allocate device memory when they call in: plugin interfaces whose enqueue step must not
 * allocate, code running while a CUDA graph is being captured (cudaMalloc is not allowed then),
 * processes whose device memory is all handed out up front by one custom allocator. The pages
 * have no counterpart: this is an interface convenience, not part of the method.
 *
 * Scratch: a fixed array of STRATA_NOALLOC_SCRATCH_BYTES in the library's device globals. Every
 * GPU that loads the library holds it until the process exits. Requests whose scratch would not
 * fit (strata_route_workspace_size(T, E, k) > STRATA_NOALLOC_SCRATCH_BYTES) return
 * STRATA_ERR_UNSUPPORTED before anything runs; everything else is identical to
 * strata_route_topk (same arguments, outputs and checks, applied in the same order, the size
 * limit last). Nothing is allocated or freed, by the library or any routine it calls.
 * Set-up: every call made while `stream` is not capturing looks up the array's device address in
 * the current context (cudaGetSymbolAddress, with the device current) and keeps it; a call made
 * while `stream` captures uses the address kept by the last uncaptured call on that device, and
 * returns STRATA_ERR_UNSUPPORTED if there was none. So make one call on each device (and again
 * after a device reset or a switch to another context) before capturing it.
 * All calls share the one array: calls that overlap on the GPU (different streams, or several
 * host threads) race and must be serialised by the caller. Each call clears the status header it
 * needs before its kernels run; the rest of the array keeps the previous call's contents.
 * Device status of the last call: strata_workspace_status is not available (no workspace
 * pointer); data faults still never trap.
 */
#define STRATA_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB per device */
strata_status strata_route_topk_noalloc(const void* x_bf16, const float* w_router,
                                        const float* bias, int64_t T, int64_t H, int32_t E,
                                        int32_t k, uint32_t flags, int32_t* ids, float* gates,
                                        int32_t* counts, int32_t* offsets, int32_t* perm,
                                        int32_t* inv, strata_stream stream);

/*
 * strata_group_rows — the grouping step alone, for routes the caller computed ([tuning-3090]
 * §3.2: the rows routed to one expert are gathered into one group of the grouped GEMM): the
 * counts, offsets, perm and inv of strata_route_topk for a given ids [T,k] int32 (device), rows
 * ordered by (expert, token, slot) (a token may name one expert in several slots).
 * counts [E], offsets [E+1] (required); perm [T*k], inv [T,k] (required when T > 0); all int32,
 * device, 4-byte aligned. An id outside [0, E) sets STRATA_DEV_BAD_ID in the workspace status
 * word; its row is left out of every group (inv = -1, no perm entry) and offsets[E] counts the
 * valid rows only, which keep the positions they would have without the invalid ones.
 * Limits: 0 <= T <= 2^22, 1 <= k <= 32, 1 <= E <= 1024. workspace >=
 * STRATA_GROUP_WORKSPACE_BYTES, 256-byte aligned (it holds the status word only).
 */
#define STRATA_GROUP_WORKSPACE_BYTES 256u
strata_status strata_group_rows(const int32_t* ids, int64_t T, int32_t k, int32_t E,
                                int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                void* workspace, size_t ws_bytes, strata_stream stream);

/*
 * One routed MoE FFN layer. Expert weights are the outputs of strata_quantize_groups, stacked
 * over experts; the shared expert, when has_shared != 0, is index E of each stack.
 * Expert e computes y = (silu(x Wg_e^T) * (x Wu_e^T)) Wd_e^T   ([glm-4090] §01: Gate/Up, Down).
 */
typedef struct {
  int64_t H;             /* hidden size, % 128 == 0 */
  int64_t I;             /* expert intermediate size, % 128 == 0 */
  int32_t E;             /* routed experts, 1..1024 */
  int32_t k;             /* experts per token, 1..min(E, 32) */
  int32_t has_shared;    /* 0 or 1: expert E is always on, gate 1 */
  uint32_t flags;        /* STRATA_RENORM | STRATA_ADD_RESIDUAL | STRATA_ROUTER_FP16 |
                            STRATA_FORCE_*_PATH | STRATA_WS_REUSE */
  const float* w_router; /* [E, H] fp32, or fp16 with STRATA_ROUTER_FP16 (cast the pointer) */
  const float* bias;     /* [E] fp32 or NULL */
  const uint8_t* gate_codes; const void* gate_scales; /* [E+S, I, H/2] u8, [E+S, I, H/128] fp16 */
  const uint8_t* up_codes;   const void* up_scales;   /* same shapes */
  const uint8_t* down_codes; const void* down_scales; /* [E+S, H, I/2] u8, [E+S, H, I/128] fp16 */
  int32_t group_size;    /* scale group of all three projections: 128 (0 means 128), 64 or 256;
                            the scales above are then [.., K/group_size]. 256 on the decode path
                            needs H % 512 == 0 and I % 512 == 0 */
  int32_t bits;          /* code width of all three projections: 4 (0 means 4) or 8. With 8 the
                            codes are int8, one per byte (strata_quantize_groups_bits): gate/up
                            [E+S, I, H], down [E+S, H, I]; such layers run on the tensor-core
                            grouped GEMM at every batch size (STRATA_FORCE_WARP_PATH ->
                            STRATA_ERR_UNSUPPORTED) */
} strata_moe_layer;

/* Workspace bytes strata_moe_forward needs for up to T_max tokens (0 if the layer is invalid). */
size_t strata_moe_workspace_size(const strata_moe_layer* layer, int64_t T_max);

/*
 * strata_moe_forward — out[t] = sum_j gates[t,j] * y_{ids[t,j]}(x_t) + has_shared * y_E(x_t)
 * (+ x_t with STRATA_ADD_RESIDUAL), summed in fp32 and rounded once to bf16.
 * x_bf16 [T,H], out_bf16 [T,H] bf16 (device; out may not alias x). T == 0 is a no-op.
 * workspace: >= strata_moe_workspace_size(layer, T) bytes, 256-byte aligned, device. The
 * workspace needs no initialisation; one workspace serves one stream at a time.
 */
strata_status strata_moe_forward(const strata_moe_layer* layer, const void* x_bf16, int64_t T,
                                 void* out_bf16, void* workspace, size_t ws_bytes,
                                 strata_stream stream);

/*
 * strata_moe_forward_padded — strata_moe_forward at a fixed maximum batch whose live token count
 * is read on the device when the call runs, so that one CUDA graph captured at T_max serves every
 * batch of 0..T_max tokens ([tuning-3090] §3.2: the grouped GEMM captured as a fixed graph node
 * at a fixed maximum batch, smaller batches padded with empty tokens; §5.2: every buffer
 * allocated before the graph is built).
 * n_tokens  device int32, 4-byte aligned: T, the live tokens, rows 0..T-1 of x. It is read by the
 *           call's first kernel, so a graph replays with whatever it holds at that point (write it
 *           with a copy in stream order before the replay).
 * x_bf16    [T_max, H] bf16 (device); rows T..T_max-1 are never read and may hold anything.
 * out_bf16  [T_max, H] bf16 (device); rows 0..T-1 get exactly what strata_moe_forward gives for
 *           those T tokens up to the order of its contraction sums (the GEMMs' schedule, and with
 *           it how a contraction is split between CTAs, is chosen for T_max); rows T..T_max-1 are
 *           not written. The padding tokens route to no expert and cost no weight traffic: every
 *           grid is sized for T_max, every loop stops at T.
 * A count outside [0, T_max] sets STRATA_DEV_BAD_TOKENS in the device status word and the call
 * then runs with no live token (out untouched).
 * T_max: 1..64 (the fused decode router); 4-bit codes; not STRATA_FORCE_TC_PATH. Otherwise
 * STRATA_ERR_UNSUPPORTED (T_max < 1: STRATA_ERR_SHAPE). workspace >=
 * strata_moe_workspace_size(layer, T_max). Other errors as strata_moe_forward.
 */
strata_status strata_moe_forward_padded(const strata_moe_layer* layer, const void* x_bf16,
                                        const int32_t* n_tokens, int64_t T_max, void* out_bf16,
                                        void* workspace, size_t ws_bytes, strata_stream stream);

/*
 * strata_moe_stack_forward — n_layers MoE layers in sequence with a residual add between them:
 *   x_0 = x,  x_{l+1} = bf16(x_l + MoE_l(x_l)),  out = x_{n_layers}
 * (each layer as strata_moe_forward with STRATA_ADD_RESIDUAL; no normalisation is applied, none
 * being named for the stack). layers: host array of n_layers descriptors (1..256), all with the
 * same H. x_bf16, out_bf16: [T,H] bf16, device, distinct. workspace >=
 * strata_moe_stack_workspace_size (device, 256-byte aligned, caller-owned; it also holds the two
 * intermediate activation buffers). The device status word at the workspace start collects the
 * STRATA_DEV_* bits of every layer (strata_workspace_status reads it after the stack). Errors:
 * as strata_moe_forward, checked for every layer before the first launch; STRATA_ERR_SHAPE when
 * the layers' H differ.
 */
size_t strata_moe_stack_workspace_size(const strata_moe_layer* layers, int32_t n_layers,
                                       int64_t T_max);
strata_status strata_moe_stack_forward(const strata_moe_layer* layers, int32_t n_layers,
                                       const void* x_bf16, int64_t T, void* out_bf16,
                                       void* workspace, size_t ws_bytes, strata_stream stream);

/*
 * strata_moe_forward_ex — strata_moe_forward that also copies the routing out (each pointer
 * optional, device): ids [T,k], gates [T,k], counts [E], offsets [E+1], perm [T*k], inv [T,k],
 * with the meanings of strata_route_topk.
 */
strata_status strata_moe_forward_ex(const strata_moe_layer* layer, const void* x_bf16, int64_t T,
                                    void* out_bf16, int32_t* ids, float* gates, int32_t* counts,
                                    int32_t* offsets, int32_t* perm, int32_t* inv,
                                    void* workspace, size_t ws_bytes, strata_stream stream);

/*
 * strata_moe_forward_stats — strata_moe_forward that also accumulates expert-activation statistics
 * (the hot-expert list of "Strata" 3090 tuning, xdnf.cn/news/329730, §5.5): expert_rows[e] +=
 * rows routed to expert e in this batch, and expert_rows[E] += T for the shared expert.
 * expert_rows: [E + has_shared] uint64, device, 8-byte aligned, caller-owned and caller-zeroed;
 * calls on several streams may accumulate into the same array (atomic adds). Results and errors
 * are those of strata_moe_forward; STRATA_ERR_INVALID_ARG if expert_rows is NULL or unaligned.
 */
strata_status strata_moe_forward_stats(const strata_moe_layer* layer, const void* x_bf16,
                                       int64_t T, void* out_bf16, uint64_t* expert_rows,
                                       void* workspace, size_t ws_bytes, strata_stream stream);

/*
 * strata_moe_forward_profiled — strata_moe_forward that also records caller-created CUDA events
 * (cudaEvent_t, passed as void*) on `stream` at the stage boundaries, for per-kernel timing:
 *   events[0] before the router, [1] after the router (logits + top-k), [2] after the grouping,
 *   [3] after the gate/up grouped GEMM, [4] after the down grouped GEMM, [5] after the combine.
 * n_events must be 6; any NULL event is skipped. Results are identical to strata_moe_forward.
 */
#define STRATA_PROFILE_EVENTS 6
strata_status strata_moe_forward_profiled(const strata_moe_layer* layer, const void* x_bf16,
                                          int64_t T, void* out_bf16, void* workspace,
                                          size_t ws_bytes, strata_stream stream,
                                          void* const* events, int32_t n_events);

/*
 * strata_moe_forward_host — the same layer with HOST activations: copies x_host (bf16 [T,H],
 * host memory, best pinned) to the workspace, runs the layer, copies the result to out_host
 * (bf16 [T,H], host). BLOCKING: returns after out_host is written (synchronizes `stream`).
 * workspace >= strata_moe_workspace_size(layer, T) + strata_moe_host_staging_size(layer, T).
 */
size_t strata_moe_host_staging_size(const strata_moe_layer* layer, int64_t T_max);
strata_status strata_moe_forward_host(const strata_moe_layer* layer, const void* x_host,
                                      int64_t T, void* out_host, void* workspace, size_t ws_bytes,
                                      strata_stream stream);

/*
 * Device status of a route/forward workspace: synchronizes `stream`, returns the status word in
 * *status_out (host) and clears it. Returns STRATA_ERR_TIMEOUT when STRATA_DEV_TIMEOUT was set (a
 * bounded device wait gave up: the call's outputs are incomplete), else STRATA_ERR_DEVICE_STATUS
 * when any other bit was set, else STRATA_OK.
 */
strata_status strata_workspace_status(void* workspace, strata_stream stream, uint32_t* status_out);

/* Same for a caller-owned device status word (e.g. the one given to strata_quantize_groups). */
strata_status strata_read_status(uint32_t* dev_status, strata_stream stream, uint32_t* status_out);

/*
 * strata_selftest_bounded_waits — a diagnostic of the failure path of the library's two bounded
 * device waits (no data path): the mbarrier wait of the TMA-fed grouped GEMMs and the counter
 * spin of the fused router run, one after the other, on a barrier and a counter that nothing
 * completes, each with a limit of limit_cycles SM clocks instead of its ~1-2 s. Each must give
 * up, OR STRATA_DEV_TIMEOUT into dev_words[0] and return, so the kernel ends after about
 * 2 * limit_cycles clocks and the context stays usable.
 * dev_words  [4] uint32, device, 16-byte aligned, caller-zeroed: [0] status word (read it with
 *            strata_read_status, which then returns STRATA_ERR_TIMEOUT), [1] the counter (must
 *            stay 0), [2] / [3] set to 1 when the mbarrier wait / the counter spin gave up.
 * limit_cycles 1 .. 4e9; outside -> STRATA_ERR_INVALID_ARG. Asynchronous on `stream`.
 */
strata_status strata_selftest_bounded_waits(uint32_t* dev_words, int64_t limit_cycles,
                                            strata_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* STRATA_H_ */
