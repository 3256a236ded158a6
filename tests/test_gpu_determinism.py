"""Bit-identity of repeated forwards on the decode path (the CTA-staged grouped GEMM).

The same layer and input must give the same output bits on every call, whatever order the
persistent CTAs claim their work items in: the split-K reductions sum in a fixed order, the
routing and grouping are deterministic, and the ring of shared-memory stages must never hand a
consumer a stage that the producer has begun to overwrite. That last property depends on the
cross-proxy fence between the consumers' generic-proxy reads and the producer's next TMA box; a
build without it gave a different output in about one forward in a hundred at the c4 shape
(T=4), so each case runs hundreds of forwards. At one token both GEMMs split the contraction
(the split-K reduction runs) on both the c2 and the c4 shapes.
"""
import numpy as np
import pytest

from helpers import bf16_tensor, build_gpu_layer
from workloads import CONFIGS, gen

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("key,T,n", [("c4", 4, 400), ("c4", 1, 200), ("c2", 1, 200),
                                     ("c2", 16, 200)])
def test_repeated_forwards_are_bit_identical(key, T, n):
    import torch
    import int4_grouped_expert_gb300 as st
    wl = CONFIGS[key]
    L = build_gpu_layer(wl)[0]
    x = bf16_tensor(gen.activations(T, wl.H, wl.seed, name=f"determinism/{T}"))
    ws = torch.empty(L.workspace_size(T), dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(x)
    st.check(st.strata_moe_forward(L.struct(), x, T, ref, ws, ws.numel()), "forward")
    outs = torch.empty((n,) + tuple(x.shape), dtype=x.dtype, device="cuda")
    for i in range(n):  # back to back on one stream and one workspace
        st.check(st.strata_moe_forward(L.struct(), x, T, outs[i], ws, ws.numel()), "forward")
    torch.cuda.synchronize()
    s, v = st.strata_workspace_status(ws)
    assert s == 0, f"device status 0x{v:x}"
    same = (outs.view(torch.int16) == ref.view(torch.int16)).reshape(n, -1).all(dim=1).cpu().numpy()
    bad = np.nonzero(~same)[0]
    assert bad.size == 0, f"{bad.size}/{n} forwards differ from the first (e.g. {bad[:8]})"
