"""fp64 NumPy oracle of the routed MoE FFN layer with int4 group-quantized experts.

TEST INFRASTRUCTURE ONLY (see the package docstring): imported by tests/,
__graft_entry__.smoke() and bench.py's CPU-baseline legs, never by the library.

Sources (five web write-ups about the "Strata" MoE engine; the pages have no
titles, so each is named by its address):
  [tuning-3090]  xdnf.cn/news/329730          hot/cold experts, grouped GEMM
  [tuning-moe]   lpnh.cn/news/2730718         group_quantize sketch (§2.1),
                                              fused top-k + softmax (§2.3)
  [tok-102]      zwxr.cn/news/276292          routing engine (§3.2)
  [glm-4090]     haowenji.com/articles/x-2109226022155796480
                                              Gate/Up + Down experts, 8 routed
                                              + 1 shared per token (§01)

Readings taken where the pages are silent:
  * quantize: round half to even (torch .round()); quotient w/s exact, from the
    scale as stored in fp16; a group whose stored scale is 0 gets codes 0;
    K % 128 != 0 is an error; non-finite weights are an error.
  * codes are packed two per byte, even k in the low nibble, 4-bit two's
    complement (the sketch keeps one int8 per code; the packing is ours).
  * route: logits = x Wr^T + b in full precision, softmax over all E experts,
    top-k by descending probability with ties to the lower expert id, gates are
    the top-k probabilities, not renormalised (renormalising is an option).
  * expert FFN: h = silu(x Wg^T) * (x Wu^T), y = h Wd^T with the exact
    dequantised weights q*s; out = sum_j gate_j y_j (+ shared expert, gate 1)
    (+ the layer input when a residual is requested).
"""
from __future__ import annotations

import numpy as np

GROUP = 128          # [tuning-moe] §2.1: 128 weights per group (the pages' choice)
GROUPS = (64, 128, 256)  # the sketch takes group_size as a parameter; 64 and 256 are the sizes
                         # the pages weighed against 128, kept as variants
BITS = (4, 8)        # [tuning-moe] §2.1: the sketch takes bits as a parameter (4 for experts;
                     # the pages keep attention projections at 8 bits)


def code_range(bits: int):
    """(qmin, qmax, divisor) of a bit width, [tuning-moe] §2.1.

    scale = absmax / (2**(bits-1) - 1); the sketch's clamp(-8, 7) is the bits = 4 instance of
    the two's-complement range [-2**(bits-1), 2**(bits-1) - 1], which is the range taken for 8.
    """
    if bits not in BITS:
        raise ValueError("bits must be 4 or 8")
    qmax = 2 ** (bits - 1) - 1
    return -(qmax + 1), qmax, float(qmax)


# ----------------------------------------------------------------------------- storage

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def pack_codes(q: np.ndarray) -> np.ndarray:
    """int codes [N, K] in [-8, 7] -> uint8 [N, K/2]; element 2m in the low nibble."""
    q = np.asarray(q)
    nib = (q.astype(np.int64) & 0xF).astype(np.uint8)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 [N, K/2] -> int8 [N, K] (4-bit two's complement nibbles)."""
    c = np.asarray(codes, dtype=np.uint8)
    lo = (c & 0xF).astype(np.int16)
    hi = (c >> 4).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty((c.shape[0], c.shape[1] * 2), dtype=np.int8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


# ----------------------------------------------------------------------------- quantize

def _check_weight(w16, group):
    w = np.asarray(w16)
    if w.dtype != np.float16 or w.ndim != 2:
        raise TypeError("weight must be a 2-D float16 array [out, in]")
    if group not in GROUPS:
        raise ValueError("group size must be 64, 128 or 256")
    if w.shape[1] % group:
        raise ValueError("in_features must be a multiple of the group size")
    if not np.all(np.isfinite(w)):
        raise ValueError("non-finite weight")
    return w


def quantize_groups(w16: np.ndarray, group: int = GROUP, bits: int = 4):
    """Symmetric group quantization, [tuning-moe] §2.1 (group_quantize sketch).

    weight [out, in] is viewed as [out, in/G, G] (G = group, 128 unless given); per group
      scale = absmax / (2**(bits-1) - 1)  (7 for 4 bits, 127 for 8), stored as fp16
              (nearest-even),
      q     = clamp(round_half_even(w / scale), qmin, qmax)  with the exact quotient.
    Returns (codes, scales float16 [out, in/G]); codes are uint8 [out, in/2] (two 4-bit codes
    per byte) for bits = 4 and int8 [out, in] (one code per byte) for bits = 8.
    """
    qmin, qmax, qdiv = code_range(bits)
    w = _check_weight(w16, group)
    n, kdim = w.shape
    wg = w.astype(np.float64).reshape(n, kdim // group, group)
    absmax = np.abs(wg).max(axis=-1)                      # exact
    # One rounding: the fp64 quotient absmax/7 (or /127) never sits on an fp16 midpoint unless
    # the exact one does (the exact quotient of an 11-bit significand by 7 or 127 is either
    # exact in fp16 or at least 2^-18 relative away from every midpoint).
    scale16 = (absmax / qdiv).astype(np.float16)
    s = scale16.astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        # fp64 quotient of two fp16 values decides every .5 tie exactly.
        r = np.where(s > 0, np.rint(wg / s), 0.0)
    q = np.clip(r, qmin, qmax).astype(np.int8).reshape(n, kdim)
    return (pack_codes(q) if bits == 4 else q), scale16


def quantize_groups_f16_quotient(w16: np.ndarray, group: int = GROUP, bits: int = 4):
    """The literal fp16 reading of the sketch: w / scale rounded to fp16 before round().

    Not the chosen reading; kept so the tests can count where the two differ.
    """
    qmin, qmax, qdiv = code_range(bits)
    w = _check_weight(w16, group)
    n, kdim = w.shape
    wg = w.reshape(n, kdim // group, group)
    absmax = np.abs(wg.astype(np.float64)).max(axis=-1)
    scale16 = (absmax / qdiv).astype(np.float16)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = (wg.astype(np.float64) / scale16.astype(np.float64)[..., None]).astype(np.float16)
        r = np.where(scale16[..., None] > 0, np.rint(quot.astype(np.float64)), 0.0)
    q = np.clip(r, qmin, qmax).astype(np.int8).reshape(n, kdim)
    return (pack_codes(q) if bits == 4 else q), scale16


def dequantize(codes: np.ndarray, scales: np.ndarray, group: int = None) -> np.ndarray:
    """q * scale in fp64, [out, in]; the group size follows from the shapes unless given.

    codes: packed 4-bit (uint8 [out, in/2]) or 8-bit (int8 [out, in]), told apart by dtype.
    """
    c = np.asarray(codes)
    q = (c if c.dtype == np.int8 else unpack_codes(c)).astype(np.float64)
    n, kdim = q.shape
    if group is None:
        group = kdim // np.asarray(scales).shape[1]
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    return (q.reshape(n, kdim // group, group) * s[..., None]).reshape(n, kdim)


# ----------------------------------------------------------------------------- route

def route_topk(x_bits: np.ndarray, w_router: np.ndarray, bias, k: int, renorm: bool = False):
    """Router softmax + top-k, [tuning-moe] §2.3 (point 1) and [tok-102] §3.2.

    logits = x Wr^T + b (fp64, x taken exactly from its bf16 bits), p = softmax
    over the E experts, ids = the k largest p in descending order (ties to the
    lower id), gates = p[ids] (renormalised over the k only when asked).
    Returns dict(ids int32 [T,k], gates f64 [T,k], probs f64 [T,E],
    gap f64 [T] = p_(k) - p_(k+1) (inf when k == E), inner_gap f64 [T] =
    smallest gap between adjacent selected probabilities, dot_l2 f64 [T,E] =
    ||x_t * w_e||_2, the size of each logit's product terms, from which the
    rounding error of a finite-precision logit is bounded).
    """
    x = bf16_to_f64(x_bits)
    wr = np.asarray(w_router, dtype=np.float32).astype(np.float64)
    T = x.shape[0]
    E = wr.shape[0]
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    logits = x @ wr.T
    if bias is not None:
        logits = logits + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    m = logits.max(axis=1, keepdims=True) if T else np.zeros((0, 1))
    ex = np.exp(logits - m)
    p = ex / ex.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")       # stable: equal p keeps lower id first
    ids = order[:, :k].astype(np.int32)
    gates = np.take_along_axis(p, ids, axis=1)
    psorted = np.take_along_axis(p, order, axis=1)
    gap = psorted[:, k - 1] - psorted[:, k] if k < E else np.full(T, np.inf)
    inner = (np.min(psorted[:, :k - 1] - psorted[:, 1:k], axis=1) if k > 1
             else np.full(T, np.inf))
    if renorm:
        gates = gates / gates.sum(axis=1, keepdims=True)
    dot_l2 = np.sqrt((x * x) @ (wr * wr).T)
    return dict(ids=ids, gates=gates, probs=p, logits=logits, gap=gap, inner_gap=inner,
                dot_l2=dot_l2)


# ----------------------------------------------------------------------------- permute

def permute(ids: np.ndarray, E: int):
    """Group the routed (token, slot) rows by expert, [tuning-3090] §3.2.

    Rows are ordered by (expert, token) ascending (a token never picks one
    expert twice, so this order is unique). Returns counts [E], offsets [E+1]
    (exclusive prefix sum), perm [T*k] (source token of each row) and
    inv [T,k] (row of each (token, slot)).
    """
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    tok = np.repeat(np.arange(T, dtype=np.int64), k)
    order = np.lexsort((tok, flat))          # last key is primary: expert, then token
    perm = tok[order].astype(np.int32)
    row = np.empty(T * k, dtype=np.int64)
    row[order] = np.arange(T * k)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return dict(counts=counts, offsets=offsets, perm=perm, inv=row.reshape(T, k).astype(np.int32))


# ----------------------------------------------------------------------------- FFN

def silu(u: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return u / (1.0 + np.exp(-u))


def expert_ffn(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray):
    """One SiLU-gated expert on fp64 rows: y = (silu(x Wg^T) * (x Wu^T)) Wd^T.

    Gate/Up + Down projections per [glm-4090] §01; the SiLU gate is the
    workload's stated expert form. w_* are dequantised fp64 weights
    ([I,H], [I,H], [H,I]).
    """
    u = x @ w_gate.T
    v = x @ w_up.T
    return (silu(u) * v) @ w_down.T


def moe_forward(x_bits, w_router, bias, k, experts, E, shared=0, renorm=False,
                residual=False, tokens=None, expert_out=None):
    """The routed MoE FFN layer in fp64.

    x_bits   bf16 bits [T, H]
    experts  callable e -> ((gate_codes, gate_scales), (up_codes, up_scales),
             (down_codes, down_scales)), e in [0, E] (E = shared expert)
    tokens   optional token indices; only these output rows are computed
             (each token's output depends on its own row alone).
    expert_out  optional {e: expert_ffn rows} computed by the caller with this
             module's quantize_groups / dequantize / expert_ffn (e.g. several
             experts at once in worker processes): for a routed expert, the
             rows routed to it in the order of np.argwhere(ids == e); for the
             shared expert E, every selected token. experts is then not used.

    out[t] = sum_j gates[t,j] * FFN_{ids[t,j]}(x_t) + shared * FFN_E(x_t)
             (+ x_t when residual), summed j = 0..k-1, then shared, then x.
    The shared expert's gate is 1: [glm-4090] §01 gives it no gate.
    """
    x_all = np.asarray(x_bits, dtype=np.uint16)
    if tokens is not None:
        x_all = x_all[np.asarray(tokens)]
    r = route_topk(x_all, w_router, bias, k, renorm=renorm)
    x = bf16_to_f64(x_all)
    T, H = x.shape
    out = np.zeros((T, H), dtype=np.float64)
    ids, gates = r["ids"], r["gates"]
    deq_cache = {}

    def deq(e):
        if e not in deq_cache:
            (gc, gs), (uc, us), (dc, ds) = experts(e)
            deq_cache.clear()
            deq_cache[e] = (dequantize(gc, gs), dequantize(uc, us), dequantize(dc, ds))
        return deq_cache[e]

    def ffn(e, rows):
        if expert_out is not None:
            return expert_out[e]
        wg, wu, wd = deq(e)
        return expert_ffn(x[rows], wg, wu, wd)

    y_routed = np.zeros((T, k, H), dtype=np.float64)
    for e in np.unique(ids):
        sel = np.argwhere(ids == e)             # (token, slot) pairs routed to e
        y_routed[sel[:, 0], sel[:, 1]] = ffn(int(e), sel[:, 0])
    for j in range(k):
        out += gates[:, j:j + 1] * y_routed[:, j]
    if shared:
        out += ffn(E, np.arange(T))
    if residual:
        out += x
    return dict(out=out, route=r)
