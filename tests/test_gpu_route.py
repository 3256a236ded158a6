"""K2 router + K3 grouping via strata_route_topk vs the oracle.

ids exact (tokens whose top-k boundary gap is <= 1e-6 in the oracle's fp64
probabilities are excluded and counted), gates rtol 1e-5, counts / offsets /
perm / inv exact. Sources: "Strata" MoE tuning notes (lpnh.cn/news/2730718)
§2.3 point 1; routing engine (zwxr.cn/news/276292) §3.2; token grouping
("Strata" 3090 tuning, xdnf.cn/news/329730, §3.2).
"""
import numpy as np
import pytest

import oracle
from helpers import bf16_tensor, compare_routing
from workloads import CONFIGS, gen

pytestmark = pytest.mark.gpu


def gpu_route(x_bits, wr, bias, k, flags=0, group=True):
    import torch
    import int4_grouped_expert_gb300 as st
    T, H = x_bits.shape
    E = wr.shape[0]
    x = bf16_tensor(x_bits) if T else torch.zeros(1, H, dtype=torch.bfloat16, device="cuda")
    wdt = np.float16 if flags & st.STRATA_ROUTER_FP16 else np.float32
    w = torch.from_numpy(np.ascontiguousarray(wr, dtype=wdt)).cuda()
    b = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).cuda()
    o = dict(ids=torch.full((max(T, 1), k), -1, dtype=torch.int32, device="cuda"),
             gates=torch.zeros(max(T, 1), k, dtype=torch.float32, device="cuda"))
    if group:
        o.update(counts=torch.full((E,), -1, dtype=torch.int32, device="cuda"),
                 offsets=torch.full((E + 1,), -1, dtype=torch.int32, device="cuda"),
                 perm=torch.full((max(T * k, 1),), -1, dtype=torch.int32, device="cuda"),
                 inv=torch.full((max(T, 1), k), -1, dtype=torch.int32, device="cuda"))
    ws_bytes = st.strata_route_workspace_size(T, E, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    rc = st.strata_route_topk(x, w, b, T, H, E, k, flags, workspace=ws, ws_bytes=ws_bytes, **o)
    st.check(rc, "strata_route_topk")
    torch.cuda.synchronize()
    s, v = st.strata_workspace_status(ws)
    assert s == 0, hex(v)
    res = {kk: vv.cpu().numpy() for kk, vv in o.items()}
    if group:
        res["perm"] = res["perm"][:T * k]
    res["ids"], res["gates"] = res["ids"][:T], res["gates"][:T]
    if group:
        res["inv"] = res["inv"][:T]
    return res


def check(x, wr, b, k, flags=0):
    E = wr.shape[0]
    ref = oracle.route_topk(x, wr, b, k, renorm=bool(flags & 1))
    g = gpu_route(x, wr, b, k, flags)
    diff, near = compare_routing(g, ref, E)
    return int(diff.sum()), int(near.sum())


@pytest.mark.parametrize("key,T", [("c1", 64), ("c2", 1), ("c2", 16), ("c3", 512), ("c4", 32),
                                   ("c5", 4096)])
def test_workload_routers(key, T):
    wl = CONFIGS[key]
    x = gen.activations(T, wl.H, wl.seed, name=f"route/{key}")
    check(x, gen.router_weight(wl), gen.router_bias(wl), wl.k)


def test_zipf_variant_of_prefill_router():
    wl = CONFIGS["c3"]
    x = gen.activations(512, wl.H, 0, name="route/c3z")
    check(x, gen.router_weight(wl), gen.router_bias(wl, 0, "zipf"), wl.k)


@pytest.mark.parametrize("T,E,k", [(1, 20, 20), (7, 20, 3), (33, 33, 1), (5, 1024, 32), (3, 1, 1)])
def test_edge_shapes(T, E, k):
    rng = np.random.default_rng(E * 7 + k)
    x = gen.f32_to_bf16_bits(rng.standard_normal((T, 256)).astype(np.float32))
    wr = (rng.standard_normal((E, 256)) * 0.05).astype(np.float32)
    check(x, wr, None, k)


def test_zero_router_ties_go_to_lowest_ids():
    x = gen.activations(9, 128, 0)
    g = gpu_route(x, np.zeros((40, 128), np.float32), None, 5)
    np.testing.assert_array_equal(g["ids"], np.tile(np.arange(5), (9, 1)))
    np.testing.assert_allclose(g["gates"], 1 / 40, rtol=1e-6)


def test_all_tokens_to_one_expert_and_empty_experts():
    x = gen.activations(50, 256, 1)
    wr = np.zeros((12, 256), np.float32)
    b = np.zeros(12, np.float32)
    b[7] = 30.0
    g = gpu_route(x, wr, b, 1)
    assert (g["ids"] == 7).all()
    assert g["counts"][7] == 50 and g["counts"].sum() == 50
    np.testing.assert_array_equal(g["perm"], np.arange(50))


def test_renorm_flag():
    wl = CONFIGS["c1"]
    x = gen.activations(64, wl.H, 0, name="route/renorm")
    check(x, gen.router_weight(wl), None, wl.k, flags=1)


def test_empty_batch():
    g = gpu_route(np.zeros((0, 128), np.uint16), np.zeros((4, 128), np.float32), None, 2)
    assert (g["counts"] == 0).all() and (g["offsets"] == 0).all()


@pytest.mark.parametrize("key,T", [("c2", 16), ("c5", 1024)])
def test_fp16_router(key, T):
    """STRATA_ROUTER_FP16: the router weights stored as fp16 (the oracle gets the same fp16
    values); logits still come from exact products summed in fp32."""
    import int4_grouped_expert_gb300 as st
    wl = CONFIGS[key]
    x = gen.activations(T, wl.H, 0, name=f"route16/{key}")
    wr16 = gen.router_weight(wl).astype(np.float16).astype(np.float32)
    check(x, wr16, gen.router_bias(wl), wl.k, flags=st.STRATA_ROUTER_FP16)
