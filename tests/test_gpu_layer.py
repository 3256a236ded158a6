"""The whole layer (strata_moe_forward) vs the oracle on decode / small workloads.

Output tolerance: relative L2 <= 5e-3 and max-abs <= 3e-2 over the compared
tokens (bf16 activations, fp32 accumulation); tokens whose top-k boundary is a
near tie (gap <= 1e-6) may route differently and are then excluded, counted.
Expert form: Gate/Up + Down ("GLM-5.3-Flash on one 4090",
haowenji.com/articles/x-2109226022155796480, §01), SiLU gate, weighted combine
plus a shared expert with gate 1.
"""
import numpy as np
import pytest

import oracle
import oracle_pool
from helpers import (OracleExperts, bf16_tensor, bf16_to_np_bits, build_gpu_layer, compare_output,
                     compare_routing, run_forward)
from workloads import CONFIGS, Workload, gen

pytestmark = pytest.mark.gpu

_CACHE = {}


def layer_for(key, layer=0, router_kind=None, flags=0):
    ck = (key, layer, router_kind, flags)
    if ck not in _CACHE:
        _CACHE.clear()
        wl = CONFIGS[key]
        _CACHE[ck] = (wl,) + build_gpu_layer(wl, layer, router_kind, flags)
    return _CACHE[ck]


def check_layer(wl, L, wr, b, x, layer=0, residual=False, renorm=False, rows=None,
                overrides=None, ties_expected=False):
    g = run_forward(L, x)
    tokens = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    experts = OracleExperts(wl, layer, overrides, group=getattr(L, "group", 128),
                            bits=getattr(L, "bits", 4))
    ref = oracle.moe_forward(x, wr, b, wl.k, experts, wl.E, wl.shared,
                             renorm=renorm, residual=residual, tokens=tokens)
    full_ref = oracle.route_topk(x, wr, b, wl.k, renorm=renorm)
    diff, _ = compare_routing(g, full_ref, wl.E, ties_expected=ties_expected)
    keep = ~diff[tokens]
    compare_output(g["out"][tokens][keep], ref["out"][keep])
    return int(diff.sum())


def test_c1_single_layer_64_tokens():
    wl, L, wr, b = layer_for("c1")
    check_layer(wl, L, wr, b, gen.activations(64, wl.H, wl.seed))


@pytest.mark.parametrize("T", [1, 7, 63, 100, 200])
def test_c1_ragged_batches(T):
    # 1..64: one-launch router + CTA-staged GEMM; 100: multi-launch router, row gather, CTA-staged
    # GEMM; 200: tensor-core GEMM
    wl, L, wr, b = layer_for("c1")
    check_layer(wl, L, wr, b, gen.activations(T, wl.H, wl.seed, name=f"ragged{T}"))


@pytest.mark.parametrize("T", [1, 4, 8, 16])
def test_c2_decode_batches(T):
    wl, L, wr, b = layer_for("c2")
    check_layer(wl, L, wr, b, gen.activations(T, wl.H, wl.seed, name=f"decode{T}"))


def test_c4_layer_decode_32():
    wl, L, wr, b = layer_for("c4", layer=3)
    check_layer(wl, L, wr, b, gen.activations(32, wl.H, wl.seed, name="c4l3"), layer=3)


def test_residual_and_renorm_flags():
    import int4_grouped_expert_gb300 as st
    wl, L, wr, b = layer_for("c1", flags=st.STRATA_ADD_RESIDUAL | st.STRATA_RENORM)
    check_layer(wl, L, wr, b, gen.activations(40, wl.H, wl.seed, name="flags"), residual=True,
                renorm=True)


SMALL = Workload("t", "edge", H=256, I=384, E=20, k=20, shared=1, batches=(5,), router="uniform")


def test_k_equals_e_with_shared_and_odd_expert_count():
    wl = SMALL
    L, wr, b = build_gpu_layer(wl)
    check_layer(wl, L, wr, b, gen.activations(5, wl.H, 3))


def test_dense_equivalence_on_gpu():
    """k = E, zero router: out = mean of the experts' FFNs + shared (checked via the oracle)."""
    wl = SMALL
    wr = np.zeros((wl.E, wl.H), np.float32)
    L, wr, b = build_gpu_layer(wl, w_router=wr)
    check_layer(wl, L, wr, b, gen.activations(9, wl.H, 4), ties_expected=True)


def test_largest_expert_count_and_top_k():
    """1023 routed experts + the shared one (the library's maximum) and k = 32, 64 tokens: 2048
    routed rows, more than the compact grouping handles, so the general grouping runs."""
    wl = Workload("tmax", "max", H=256, I=128, E=1023, k=32, shared=1, batches=(64,),
                  router="uniform")
    L, wr, b = build_gpu_layer(wl)
    check_layer(wl, L, wr, b, gen.activations(64, wl.H, 11), rows=[0, 1, 31, 63])


def test_all_tokens_one_expert():
    wl = Workload("t1", "one", H=512, I=256, E=12, k=1, shared=0, batches=(70,), router="uniform")
    bias = np.zeros(wl.E, np.float32)
    bias[5] = 40.0
    L, wr, b = build_gpu_layer(wl, bias=bias)
    x = gen.activations(70, wl.H, 5)
    g = run_forward(L, x)
    assert (g["ids"] == 5).all() and g["counts"][5] == 70
    check_layer(wl, L, wr, b, x)


def test_host_entry_point_matches_device_entry_point():
    import torch
    import int4_grouped_expert_gb300 as st
    wl, L, wr, b = layer_for("c1")
    x = gen.activations(33, wl.H, 9)
    g = run_forward(L, x, taps=False)
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    s = L.struct()
    need = st.strata_moe_workspace_size(s, 33) + st.strata_moe_host_staging_size(s, 33)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st.check(st.strata_moe_forward_host(s, xh, 33, oh, ws, need), "forward_host")
    np.testing.assert_array_equal(oh.numpy().view(np.uint16), g["out"])


def test_workspace_reuse_and_determinism():
    import torch
    wl, L, wr, b = layer_for("c1")
    x = gen.activations(64, wl.H, 11)
    ws = torch.full((L.workspace_size(64),), 0x5A, dtype=torch.uint8, device="cuda")
    a = run_forward(L, x, workspace=ws)
    c = run_forward(L, gen.activations(3, wl.H, 12), workspace=ws)
    d = run_forward(L, x, workspace=ws)
    np.testing.assert_array_equal(a["out"], d["out"])
    assert c["out"].shape == (3, wl.H)


def test_forward_argument_errors():
    import torch
    import int4_grouped_expert_gb300 as st
    wl, L, wr, b = layer_for("c1")
    s = L.struct()
    x = bf16_tensor(gen.activations(4, wl.H, 0))
    out = torch.empty_like(x)
    need = L.workspace_size(4)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert st.strata_moe_forward(s, x, 4, out, ws, need - 1) == 4          # WORKSPACE
    assert st.strata_moe_forward(s, x, 4, x, ws, need) == 1                # out aliases x
    assert st.strata_moe_forward(s, x, 0, out, ws, need) == 0              # empty batch
    s.k = 17
    assert st.strata_moe_forward(s, x, 4, out, ws, need) == 1              # k > E


@pytest.mark.parametrize("T,path", [(64, "tc"), (200, "warp"), (200, "tc"), (1, "tc"), (300, "tc")])
def test_c1_both_gemm_paths(T, path):
    """The warp (mma.sync) and tensor-core (tcgen05) grouped GEMMs on the same layer."""
    import int4_grouped_expert_gb300 as st
    flag = st.STRATA_FORCE_TC_PATH if path == "tc" else st.STRATA_FORCE_WARP_PATH
    wl, L, wr, b = layer_for("c1", flags=flag)
    check_layer(wl, L, wr, b, gen.activations(T, wl.H, wl.seed, name=f"path{T}"))


def test_tc_path_shared_expert_and_long_segments():
    """Shared expert with T rows spans several 256-row tiles; k = E keeps every expert busy."""
    import int4_grouped_expert_gb300 as st
    wl = Workload("t2", "tc-edge", H=384, I=256, E=6, k=6, shared=1, batches=(600,), router="uniform")
    L, wr, b = build_gpu_layer(wl, flags=st.STRATA_FORCE_TC_PATH)
    check_layer(wl, L, wr, b, gen.activations(600, wl.H, 8))


@pytest.mark.parametrize("key,T", [("c2", 1), ("c2", 16), ("c1", 64), ("c1", 200)])
def test_workspace_reuse_flag(key, T):
    """STRATA_WS_REUSE: on a zero-filled workspace the calls skip the clearing of its header and
    give the default call's bits, call after call (the fused router resets its counters as it
    ends); the status word is not cleared per call but stays 0 here. 200 tokens take the
    multi-launch router and the tensor-core GEMMs."""
    import torch
    import int4_grouped_expert_gb300 as st
    wl, L, wr, b = layer_for(key)
    xb = gen.activations(T, wl.H, wl.seed, name=f"reuse/{T}")
    ref = run_forward(L, xb, taps=False)["out"]
    s = L.struct()
    s.flags |= st.STRATA_WS_REUSE
    x = bf16_tensor(xb)
    ws = torch.zeros(L.workspace_size(T), dtype=torch.uint8, device="cuda")
    outs = torch.empty((6, T, wl.H), dtype=torch.bfloat16, device="cuda")
    for i in range(6):
        st.check(st.strata_moe_forward(s, x, T, outs[i], ws, ws.numel()), "forward")
    torch.cuda.synchronize()
    for i in range(6):
        np.testing.assert_array_equal(bf16_to_np_bits(outs[i]), ref)
    assert st.strata_workspace_status(ws) == (0, 0)


def test_expert_statistics_accumulate_across_calls():
    """strata_moe_forward_stats adds each batch's routed rows per expert (and T for the shared
    expert) into a caller-owned counter array (the per-expert activation counts of "Strata" 3090
    tuning, xdnf.cn/news/329730, §5.5). The totals must equal the counts of the oracle's routing
    (oracle.route_topk -> oracle.permute) summed over the batches; the output equals
    strata_moe_forward's."""
    import torch
    import int4_grouped_expert_gb300 as st
    wl, L, wr, b = layer_for("c2")
    hits = torch.zeros(wl.E + wl.shared, dtype=torch.int64, device="cuda")
    expect = np.zeros(wl.E + wl.shared, np.int64)
    for T, name in ((16, "stats16"), (5, "stats5"), (64, "stats64"), (200, "stats200")):
        xb = gen.activations(T, wl.H, wl.seed, name=name)
        x = bf16_tensor(xb)
        out = torch.empty_like(x)
        ws = torch.empty(L.workspace_size(T), dtype=torch.uint8, device="cuda")
        st.check(st.strata_moe_forward_stats(L.struct(), x, T, out, hits, ws, ws.numel()), "stats")
        ref = run_forward(L, xb, taps=True)
        np.testing.assert_array_equal(bf16_to_np_bits(out), ref["out"])
        route = oracle.route_topk(xb, wr, b, wl.k)
        compare_routing(ref, route, wl.E)
        assert (ref["ids"] == route["ids"]).all(), "a near-tie token routed differently"
        expect[:wl.E] += oracle.permute(route["ids"], wl.E)["counts"]
        expect[wl.E] += T
    np.testing.assert_array_equal(hits.cpu().numpy(), expect)


def test_forward_replays_from_a_cuda_graph():
    """The forward captured once in a CUDA graph (fixed buffers, PDL chain inside) and replayed on
    new inputs copied into the captured input buffer gives the direct call's results, and matches
    the oracle."""
    import torch
    import int4_grouped_expert_gb300 as st
    wl, L, wr, b = layer_for("c2")
    T = 8
    x_static = torch.empty(T, wl.H, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x_static)
    ws = torch.empty(L.workspace_size(T), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    x_static.copy_(bf16_tensor(gen.activations(T, wl.H, wl.seed, name="graph0")))
    with torch.cuda.stream(side):  # first call outside the capture (one-time host set-up)
        st.check(st.strata_moe_forward(L.struct(), x_static, T, out, ws, ws.numel(), side), "fwd")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s = torch.cuda.current_stream()
        st.check(st.strata_moe_forward(L.struct(), x_static, T, out, ws, ws.numel(), s), "capture")
    for name in ("graph1", "graph2"):
        xb = gen.activations(T, wl.H, wl.seed, name=name)
        x_static.copy_(bf16_tensor(xb))
        g.replay()
        torch.cuda.synchronize()
        got = bf16_to_np_bits(out)
        ref = run_forward(L, xb)
        np.testing.assert_array_equal(got, ref["out"])
        diff, _ = compare_routing(ref, oracle.route_topk(xb, wr, b, wl.k), wl.E)
        rows = np.array([t for t in range(T) if not diff[t]], dtype=np.int64)
        compare_output(got[rows], oracle_pool.moe_forward(wl, xb, wr, b, rows)["out"])


@pytest.mark.parametrize("T", [16, 200])
def test_fp16_router_layer(T):
    """A layer whose router weights are stored as fp16: 16 tokens take the one-launch decode
    router, 200 the tensor-core router and GEMMs."""
    wl = CONFIGS["c1"]
    wr16 = gen.router_weight(wl).astype(np.float16).astype(np.float32)
    L, _, b = build_gpu_layer(wl, w_router=wr16)
    L.set_router(wr16, b, fp16=True)
    check_layer(wl, L, wr16, b, gen.activations(T, wl.H, wl.seed, name=f"r16_{T}"))


@pytest.mark.parametrize("group", [64, 256])
@pytest.mark.parametrize("T", [16, 100, 200])
def test_other_group_sizes(group, T):
    """Experts quantized with 64- or 256-wide groups (codes and scales from the device kernel,
    bit-exact vs the oracle), the forward on the decode path (16: one-launch router; 100:
    multi-launch router) and the tensor-core path (200)."""
    wl = CONFIGS["c1"]
    L, wr, b = build_gpu_layer(wl, group=group)
    check_layer(wl, L, wr, b, gen.activations(T, wl.H, wl.seed, name=f"g{group}_{T}"))


@pytest.mark.parametrize("group,T", [(128, 1), (128, 16), (128, 63), (128, 100), (128, 200),
                                     (64, 16), (64, 200), (256, 16), (256, 200)])
def test_8bit_experts(group, T):
    """Experts with 8-bit codes (one per byte, bit-exact vs the oracle's 8-bit quantizer) on the
    tensor-core kernel's 8-bit dequant, with the one-launch decode router (T <= 64) and the
    multi-launch router (100, 200)."""
    wl = CONFIGS["c1"]
    L, wr, b = build_gpu_layer(wl, group=group, bits=8)
    check_layer(wl, L, wr, b, gen.activations(T, wl.H, wl.seed, name=f"b8_{group}_{T}"))


def test_8bit_experts_decode_layer():
    """8-bit experts at the headline decode shape (H4096 I1536, 288 experts top-8 + shared), T=16."""
    wl = CONFIGS["c2"]
    L, wr, b = build_gpu_layer(wl, bits=8)
    check_layer(wl, L, wr, b, gen.activations(16, wl.H, wl.seed, name="b8_c2"))


def test_8bit_layer_odd_group_counts_and_forced_warp_path():
    """8-bit codes run on the tensor-core kernel at any shape (here H/128 = 3, a count the decode
    kernel cannot take); forcing the warp path is refused."""
    import int4_grouped_expert_gb300 as st
    torch = __import__("torch")
    wl = Workload("odd8", "odd-groups", H=384, I=256, E=4, k=2, shared=0, batches=(4,),
                  router="uniform")
    L, wr, b = build_gpu_layer(wl, bits=8)
    check_layer(wl, L, wr, b, gen.activations(4, wl.H, 1, name="odd8"))
    L.flags |= st.STRATA_FORCE_WARP_PATH
    x = bf16_tensor(gen.activations(4, wl.H, 1, name="odd8"))
    out = torch.empty_like(x)
    ws = torch.empty(L.workspace_size(4), dtype=torch.uint8, device="cuda")
    assert st.strata_moe_forward(L.struct(), x, 4, out, ws, ws.numel()) == 3   # UNSUPPORTED


@pytest.mark.parametrize("bits", [4, 8])
def test_tc_small_tiles_partial_code_slot(bits):
    """The 64-row tensor-core tiles (few rows per expert) with a contraction of 6 stages: 4-bit
    code slots hold 4 stages, so the second slot of each row is half past the row end (zero
    fill); 8-bit slots hold 2."""
    wl = Workload("slot", "partial-slot", H=384, I=256, E=16, k=2, shared=1, batches=(200,),
                  router="uniform")
    L, wr, b = build_gpu_layer(wl, bits=bits)
    check_layer(wl, L, wr, b, gen.activations(200, wl.H, 3, name=f"slot{bits}"))
