"""The 8-layer decode stack (hidden 4096, expert inter 2048, 128 experts top-4 + shared, Zipf
router per layer, residual add between layers): strata_moe_stack_forward against the layer-by-layer
calls, and each checked layer against the oracle, teacher-forced (the oracle's layer l takes the
GPU's bf16 input to layer l, so a sub-tolerance difference cannot flip a route in a later layer).
"""
import numpy as np
import pytest

import oracle
from helpers import OracleExperts, bf16_tensor, bf16_to_np_bits, build_gpu_layer, compare_output
from workloads import CONFIGS, gen

pytestmark = pytest.mark.gpu


def test_c4_stack_layerwise_teacher_forced():
    import torch
    import int4_grouped_expert_gb300 as st
    wl = CONFIGS["c4"]
    T = 4
    layers, routers = [], []
    for l in range(wl.layers):
        L, wr, b = build_gpu_layer(wl, layer=l, flags=st.STRATA_ADD_RESIDUAL)
        layers.append(L)
        routers.append((wr, b))
    x0 = gen.activations(T, wl.H, wl.seed, name="stack")
    x = bf16_tensor(x0)
    # layer by layer
    acts = [x0]
    cur = x
    for L in layers:
        out = torch.empty_like(cur)
        ws = torch.empty(L.workspace_size(T), dtype=torch.uint8, device="cuda")
        st.check(st.strata_moe_forward(L.struct(), cur, T, out, ws, ws.numel()), "forward")
        acts.append(bf16_to_np_bits(out))
        cur = out
    # one stack call
    structs = [L.struct() for L in layers]
    need = st.strata_moe_stack_workspace_size(structs, T)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(x)
    st.check(st.strata_moe_stack_forward(structs, x, T, out, ws, need), "stack")
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_to_np_bits(out), acts[-1])
    # teacher-forced oracle on sampled layers and tokens
    for l in (0, 3, 7):
        wr, b = routers[l]
        rows = [0, 3]
        ref = oracle.moe_forward(acts[l], wr, b, wl.k, OracleExperts(wl, l), wl.E, wl.shared,
                                 residual=True, tokens=rows)
        route = oracle.route_topk(acts[l][rows], wr, b, wl.k)
        ok = route["gap"] > 1e-6
        compare_output(acts[l + 1][rows][ok], ref["out"][ok], scale_max_abs=True)
