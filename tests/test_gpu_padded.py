"""A fixed maximum batch under one captured CUDA graph (strata_moe_forward_padded): the grouped
GEMMs captured as fixed graph nodes at a maximum batch, smaller batches padded with empty tokens
("Strata" 3090 tuning, xdnf.cn/news/329730, §3.2; its §4.3 table lists "CUDA Graph + grouped
GEMM" as the last step of the ladder).

One graph is captured at T_max = 16 on the decode layer (hidden 4096, 288 experts top-8 + shared)
and replayed with 1, 5, 16 and 0 live tokens written to the device count; a second one at T_max = 4
(where the decode GEMMs cut their stages into equal ranges per CTA) with 1, 3, 4 and 0. Rows of x
beyond the live tokens hold NaN (they must never be read), rows of out beyond them hold a sentinel
(they must not be written). Live rows are compared with the oracle; at T = T_max the padded call
must equal the unpadded one bit for bit (same launch configuration).
"""
import numpy as np
import pytest

import oracle
import oracle_pool
from helpers import bf16_tensor, bf16_to_np_bits, build_gpu_layer, compare_output, compare_routing, run_forward
from workloads import CONFIGS, gen

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC0
SENTINEL = 0x1234


@pytest.fixture(scope="module")
def layer_c2():
    wl = CONFIGS["c2"]
    return (wl,) + tuple(build_gpu_layer(wl))


def capture(layer, T_MAX):
    """The padded forward at T_MAX, captured once in a CUDA graph."""
    import torch
    import int4_grouped_expert_gb300 as st
    wl, L, wr, b = layer
    x_static = torch.zeros(T_MAX, wl.H, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    out = torch.empty_like(x_static)
    n_tok = torch.full((1,), T_MAX, dtype=torch.int32, device="cuda")
    ws = torch.empty(L.workspace_size(T_MAX), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):  # one call outside the capture (one-time host set-up)
        st.check(st.strata_moe_forward_padded(L.struct(), x_static, n_tok, T_MAX, out, ws,
                                              ws.numel(), side), "padded")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st.check(st.strata_moe_forward_padded(L.struct(), x_static, n_tok, T_MAX, out, ws,
                                              ws.numel(), torch.cuda.current_stream()), "capture")
    return wl, L, wr, b, g, x_static, out, n_tok, ws


@pytest.fixture(scope="module")
def captured16(layer_c2):
    return capture(layer_c2, 16)


@pytest.fixture(scope="module")
def captured4(layer_c2):
    return capture(layer_c2, 4)


def replay(cap, live_bits, count):
    """Write the live rows (NaN padding) and the count, replay the graph, return out's bits."""
    import torch
    import int4_grouped_expert_gb300 as st
    wl, L, wr, b, g, x_static, out, n_tok, ws = cap
    xs = np.full((x_static.shape[0], wl.H), NAN_BF16, dtype=np.uint16)
    xs[:live_bits.shape[0]] = live_bits
    x_static.copy_(bf16_tensor(xs))
    n_tok.fill_(count)
    out.view(torch.int16).fill_(SENTINEL)
    g.replay()
    torch.cuda.synchronize()
    return bf16_to_np_bits(out), st.strata_workspace_status(ws)


@pytest.mark.parametrize("T_MAX,T", [(16, 1), (16, 5), (16, 16), (16, 0),
                                     (4, 1), (4, 3), (4, 4), (4, 0)])
def test_one_graph_serves_every_batch_up_to_the_maximum(request, T_MAX, T):
    captured = request.getfixturevalue(f"captured{T_MAX}")
    wl, L, wr, b = captured[:4]
    xb = gen.activations(max(T, 1), wl.H, wl.seed, name=f"padded/{T}")[:T]
    got, (s, v) = replay(captured, xb, T)
    assert s == 0, f"device status 0x{v:x}"
    assert (got[T:] == SENTINEL).all(), "a padding row of out was written"
    if T == 0:
        return
    direct = run_forward(L, xb)           # the unpadded call on the live tokens alone
    if T == T_MAX:
        np.testing.assert_array_equal(got, direct["out"])
    diff, _ = compare_routing(direct, oracle.route_topk(xb, wr, b, wl.k), wl.E)
    rows = np.array([t for t in range(T) if not diff[t]], dtype=np.int64)
    compare_output(got[rows], oracle_pool.moe_forward(wl, xb, wr, b, rows)["out"])


@pytest.mark.parametrize("count", [17, -1])
def test_a_count_beyond_the_maximum_runs_no_token(captured16, count):
    import int4_grouped_expert_gb300 as st
    captured = captured16
    wl = captured[0]
    xb = gen.activations(16, wl.H, wl.seed, name="padded/bad")
    got, (s, v) = replay(captured, xb, count)
    assert s == st.STRATA_ERR_DEVICE_STATUS
    assert v == st.STRATA_DEV_BAD_TOKENS, f"device status 0x{v:x}"
    assert (got == SENTINEL).all()
    # the graph is still good for a valid count afterwards
    got, (s, v) = replay(captured, xb[:3], 3)
    assert s == 0 and (got[3:] == SENTINEL).all() and not (got[:3] == SENTINEL).all()
