"""Shared helpers of the GPU parity tests: build a layer from the seeded workloads, run it through the
C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np

import oracle
from workloads import CONFIGS, gen

REL_L2_TOL = 5e-3     # layer output: relative L2 over the compared rows
MAX_ABS_TOL = 3e-2    # layer output: max absolute error
TIE_GAP = 1e-6        # top-k boundary gap (oracle fp64 probabilities) below which ids may differ
GATE_RTOL = 1e-5


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


def compare_routing(gpu, ref_route, E):
    """ids exact except near-tie tokens; gates rtol; returns (mismatched tokens, near-tie tokens)."""
    ids_ref, gates_ref = ref_route["ids"], ref_route["gates"]
    gap = np.minimum(ref_route["gap"], ref_route["inner_gap"])
    diff = np.any(gpu["ids"] != ids_ref, axis=1)
    near = gap <= TIE_GAP
    bad = diff & ~near
    assert not bad.any(), f"ids differ on {bad.sum()} tokens without a near tie: {np.nonzero(bad)[0][:8]}"
    ok = ~diff
    np.testing.assert_allclose(gpu["gates"][ok], gates_ref[ok], rtol=GATE_RTOL, atol=0)
    # grouping: deterministic function of the ids the GPU chose
    p = oracle.permute(gpu["ids"], E)
    for key in ("counts", "offsets", "perm", "inv"):
        np.testing.assert_array_equal(gpu[key], p[key], err_msg=key)
    return diff, near


def compare_output(out_bits, ref_out, rows=None, scale_max_abs=False):
    """Relative L2 and max-abs error of bf16 outputs against the oracle's fp64 outputs.

    The max-abs bound is stated for N(0,1)-scale activations. With scale_max_abs it is multiplied
    by max(1, rms of the reference): a residual stream with no normalisation grows layer after
    layer, and the final bf16 rounding alone then errs by up to half an ulp of that magnitude."""
    o = gen.bf16_bits_to_f32(out_bits).astype(np.float64)
    if rows is not None:
        o, ref_out = o[rows], ref_out[rows]
    err = o - ref_out
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref_out), 1e-30)
    mx = np.abs(err).max() if err.size else 0.0
    tol = MAX_ABS_TOL
    if scale_max_abs and ref_out.size:
        tol *= max(1.0, float(np.sqrt(np.mean(ref_out ** 2))))
    assert rel <= REL_L2_TOL, f"relative L2 {rel:.3e}"
    assert mx <= tol, f"max abs {mx:.3e} > {tol:.3e}"
    return rel, mx


def config(key):
    return CONFIGS[key]
