"""Shared helpers of the GPU parity tests: build a layer from the seeded workloads, run it through the
C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np

import oracle
from workloads import CONFIGS, gen

REL_L2_TOL = 5e-3     # layer output: relative L2 over the compared rows
MAX_ABS_TOL = 3e-2    # layer output: max absolute error
TIE_GAP = 1e-6        # top-k boundary gap (oracle fp64 probabilities) below which ids may differ
GATE_RTOL = 1e-5      # gate tolerance floor; see gate_rtol
U32 = 2.0 ** -24      # fp32 unit roundoff
FP32_MIN_NORMAL = 2.0 ** -126


def gate_rtol(route):
    """Relative tolerance of each token's gates: no bound is stated for them, so it follows from
    the arithmetic. A logit summed in fp32 from rounded products errs by about u * ||x_t * w_e||_2
    (random rounding errors; ten times that is the bound taken per logit). A gate is
    exp(l_j - m) / sum_e exp(l_e - m): its relative error is the error of l_j minus the
    probability-weighted mean of the errors of all l_e, so up to twice the logit bound. Never
    below GATE_RTOL: 1e-5 for N(0,1) activations, wider only where the activations are large
    (deep layers of a residual stack without normalisation)."""
    return np.maximum(GATE_RTOL, 2 * 10 * U32 * route["dot_l2"].max(axis=1))


def torch_mod():
    import torch
    return torch


def bf16_tensor(bits: np.ndarray, device="cuda"):
    torch = torch_mod()
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)


def bf16_to_np_bits(t) -> np.ndarray:
    torch = torch_mod()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


class OracleExperts:
    """Oracle-side expert provider: regenerate the fp16 weights, quantize with the oracle."""

    def __init__(self, wl, layer=0, overrides=None, group=128, bits=4):
        self.wl, self.layer, self.group, self.bits = wl, layer, group, bits
        self.cache = {}
        self.overrides = overrides or {}

    def fp16(self, e):
        if e in self.overrides:
            return self.overrides[e]
        return gen.expert_weights(self.wl, e, self.layer)

    def __call__(self, e):
        if e not in self.cache:
            if len(self.cache) > 4:
                self.cache.clear()
            self.cache[e] = tuple(oracle.quantize_groups(m, group=self.group, bits=self.bits)
                                  for m in self.fp16(e))
        return self.cache[e]


def build_gpu_layer(wl, layer=0, router_kind=None, flags=0, bias=None, w_router=None,
                    overrides=None, threads=0, experts=None, group=128, bits=4):
    """MoELayer with the workload's router and experts, quantized on the device."""
    from int4_grouped_expert_gb300 import MoELayer
    torch = torch_mod()
    L = MoELayer(wl.H, wl.I, wl.E, wl.k, wl.shared, flags=flags, group=group, bits=bits)
    wr = gen.router_weight(wl, layer) if w_router is None else w_router
    b = gen.router_bias(wl, layer, router_kind) if bias is None else bias
    L.set_router(wr, b)
    n = wl.E + wl.shared
    overrides = overrides or {}
    batch = 16
    for s in range(0, n, batch):
        es = list(range(s, min(n, s + batch)))
        if experts is not None:                 # only these experts get weights (others stay 0)
            es = [e for e in es if e in experts]
        todo = [e for e in es if e not in overrides]
        mats = dict(zip(todo, gen.expert_weights_many(wl, todo, layer, threads)))
        mats.update({e: overrides[e] for e in es if e in overrides})
        for e in es:
            L.load_expert_fp16(e, *mats[e])
    torch.cuda.synchronize()
    L.check_status()
    return L, wr, b


def run_forward(L, x_bits, workspace=None, taps=True):
    import int4_grouped_expert_gb300 as st
    torch = torch_mod()
    T = x_bits.shape[0]
    x = bf16_tensor(x_bits)
    out = torch.empty_like(x)
    ws_bytes = L.workspace_size(T)
    ws = workspace if workspace is not None else torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    E, k = L.E, L.k
    t = dict(ids=torch.empty(T, k, dtype=torch.int32, device="cuda"),
             gates=torch.empty(T, k, dtype=torch.float32, device="cuda"),
             counts=torch.empty(E, dtype=torch.int32, device="cuda"),
             offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
             perm=torch.empty(T * k, dtype=torch.int32, device="cuda"),
             inv=torch.empty(T, k, dtype=torch.int32, device="cuda"))
    if taps:
        rc = st.strata_moe_forward_ex(L.struct(), x, T, out, workspace=ws, ws_bytes=ws_bytes, **t)
    else:
        rc = st.strata_moe_forward(L.struct(), x, T, out, ws, ws_bytes)
    st.check(rc, "strata_moe_forward")
    torch.cuda.synchronize()
    s, v = st.strata_workspace_status(ws)
    assert s == 0, f"device status 0x{v:x}"
    res = {kk: vv.cpu().numpy() for kk, vv in t.items()}
    res["out"] = bf16_to_np_bits(out)
    return res


MAX_NEAR_TIE_FRAC = 0.01   # near-tie tokens allowed before the comparison is considered too weak


def compare_routing(gpu, ref_route, E, ties_expected=False):
    """ids exact except at near ties; gates within gate_rtol; grouping exact (of the GPU's ids).

    Returns (material, near): near marks tokens with a near tie (top-k boundary, or an adjacent
    pair inside the top k, closer than TIE_GAP in the oracle's fp64 probabilities); material marks
    tokens whose ids differ in a way the output can see: the selected set differs and a swapped
    expert has probability above TIE_GAP. A different order inside the top k, or a swap between
    experts of probability <= TIE_GAP (deep layers of a residual stack, where the tail of the
    softmax is ~1e-20), leaves the output as it is, so such tokens stay in the output comparison.
    Material near-tie differences are excluded from the output check and counted: the count is
    printed and bounded, so that a router that broke ties everywhere could not pass quietly
    (ties_expected: a test that builds ties on purpose, e.g. a zero router). Ids that differ
    without a near tie fail."""
    ids_ref, gates_ref = ref_route["ids"], ref_route["gates"]
    gap = np.minimum(ref_route["gap"], ref_route["inner_gap"])
    diff = np.any(gpu["ids"] != ids_ref, axis=1)
    near = gap <= TIE_GAP
    T = len(near)
    material = np.zeros(T, dtype=bool)
    for t in np.nonzero(diff)[0]:
        swapped = set(gpu["ids"][t].tolist()) ^ set(ids_ref[t].tolist())
        material[t] = any(ref_route["probs"][t, e] > TIE_GAP for e in swapped)
    print(f"routing: {T} tokens, {int(near.sum())} with a near tie (gap <= {TIE_GAP:g}); "
          f"{int((diff & near).sum())} of them routed differently, {int((material & near).sum())} "
          f"of those in a way the output sees (excluded from the output check)")
    if not ties_expected:
        assert (material & near).sum() <= max(1, int(MAX_NEAR_TIE_FRAC * T)), \
            f"{(material & near).sum()} excluded of {T}"
    bad = diff & ~near
    assert not bad.any(), f"ids differ on {bad.sum()} tokens without a near tie: {np.nonzero(bad)[0][:8]}"
    ok = ~diff
    rtol = gate_rtol(ref_route)[ok][:, None]
    # gates below the smallest normal fp32 value underflow to subnormals or zero in fp32
    err = np.abs(gpu["gates"][ok] - gates_ref[ok])
    lim = rtol * np.abs(gates_ref[ok]) + FP32_MIN_NORMAL
    worst = np.unravel_index(np.argmax(err / lim), err.shape) if err.size else None
    assert (err <= lim).all(), (f"gates differ: {gpu['gates'][ok][worst]:.6e} vs "
                                f"{gates_ref[ok][worst]:.6e}, allowed {lim[worst]:.3e}")
    # grouping: deterministic function of the ids the GPU chose
    p = oracle.permute(gpu["ids"], E)
    for key in ("counts", "offsets", "perm", "inv"):
        np.testing.assert_array_equal(gpu[key], p[key], err_msg=key)
    return material, near


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 values (8 significant bits) at |v| (normal range; 0 at 0)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(a)                       # a = m * 2**e, m in [0.5, 1)
    return np.where(a > 0, np.ldexp(1.0, e - 9), 0.0)


def compare_output(out_bits, ref_out, rows=None, scale_max_abs=False):
    """Relative L2 and max-abs error of bf16 outputs against the oracle's fp64 outputs.

    The max-abs bound (3e-2, for bf16 activations with fp32 accumulation) applies to the error of
    the arithmetic: the output's final rounding to bf16 adds up to half an ulp of the element
    (0.031 for entries in [8, 16)), which no bf16-producing implementation avoids, so it is
    allowed on top: |out - ref| - half_ulp(out) <= bound. The raw max-abs is printed beside it.
    With scale_max_abs the bound is multiplied by max(1, rms of the reference): a residual stream
    with no normalisation grows layer after layer, and relative errors grow with it."""
    o = gen.bf16_bits_to_f32(out_bits).astype(np.float64)
    if rows is not None:
        o, ref_out = o[rows], ref_out[rows]
    err = o - ref_out
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref_out), 1e-30)
    raw = np.abs(err).max() if err.size else 0.0
    mx = np.maximum(np.abs(err) - bf16_half_ulp(o), 0.0).max() if err.size else 0.0
    tol = MAX_ABS_TOL
    if scale_max_abs and ref_out.size:
        tol *= max(1.0, float(np.sqrt(np.mean(ref_out ** 2))))
    print(f"output: {o.shape[0]} rows, relative L2 {rel:.3e} (bound {REL_L2_TOL:g}), max abs "
          f"{raw:.3e}, beyond the output's bf16 rounding {mx:.3e} (bound {tol:.3e}"
          f"{', scaled by the output rms' if tol != MAX_ABS_TOL else ''})")
    if err.size:
        i = np.unravel_index(np.argmax(np.abs(err)), err.shape)
        big = np.abs(ref_out) >= 8
        print(f"        worst element: reference {ref_out[i]:.5f}, got {o[i]:.5f}; "
              f"{int(big.sum())} of {ref_out.size} reference entries are >= 8 in magnitude "
              f"(bf16 half-ulp there >= {2.0 ** -5:g}); rms of the reference "
              f"{np.sqrt(np.mean(ref_out ** 2)):.3f}")
    assert rel <= REL_L2_TOL, f"relative L2 {rel:.3e}"
    assert mx <= tol, f"max abs {mx:.3e} > {tol:.3e}"
    return rel, mx


def config(key):
    return CONFIGS[key]
