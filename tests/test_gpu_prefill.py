"""Prefill workloads on the tensor-core path vs the oracle, at full size.

c3: 512 tokens, hidden 5120, expert inter 2048, 64 experts top-4 (uniform router and a Zipf
variant). c5: 4096 tokens, hidden 7168, expert inter 2048, 256 experts top-8 + shared, fp16
experts quantized on the device first. Routing, grouping and quantization are compared in full;
the layer output on a seeded token sample (each token's output depends only on its own row, so
the oracle computes just those tokens' experts, in worker processes: tests/oracle_pool.py). The
c5 sample adds the tokens whose rows end the shared expert's segment (its last 256-row tile) and
the rows ending the largest and the smallest routed segments (their tail tiles).
"""
import numpy as np
import pytest

import oracle
import oracle_pool
from helpers import build_gpu_layer, compare_output, compare_routing, run_forward
from workloads import CONFIGS, gen

pytestmark = pytest.mark.gpu


def sample_tokens(T, n, seed):
    return np.sort(np.random.default_rng(seed).choice(T, n, replace=False))


@pytest.mark.parametrize("router", ["uniform", "zipf"])
def test_c3_prefill(router):
    wl = CONFIGS["c3"]
    L, wr, b = build_gpu_layer(wl, router_kind=router)
    x = gen.activations(512, wl.H, wl.seed, name=f"c3/{router}")
    g = run_forward(L, x)
    ref_route = oracle.route_topk(x, wr, b, wl.k)
    diff, _ = compare_routing(g, ref_route, wl.E)
    rows = np.array([t for t in sample_tokens(512, 128, 3) if not diff[t]], dtype=np.int64)
    ref = oracle_pool.moe_forward(wl, x, wr, b, rows)
    compare_output(g["out"][rows], ref["out"])


def test_c5_quantize_then_prefill():
    import torch
    wl = CONFIGS["c5"]
    L, wr, b = build_gpu_layer(wl)
    # device quantization vs the oracle on a sample of experts (all three matrices)
    for e in (0, 131, wl.E):
        mats = gen.expert_weights(wl, e)
        gpu = [(L.gate_codes[e], L.gate_scales[e]), (L.up_codes[e], L.up_scales[e]),
               (L.down_codes[e], L.down_scales[e])]
        for m, (c, s) in zip(mats, gpu):
            rc, rs = oracle.quantize_groups(m)
            np.testing.assert_array_equal(c.cpu().numpy(), rc)
            np.testing.assert_array_equal(s.cpu().numpy().view(np.uint16), rs.view(np.uint16))
    x = gen.activations(4096, wl.H, wl.seed, name="c5")
    g = run_forward(L, x)
    ref_route = oracle.route_topk(x, wr, b, wl.k)
    diff, _ = compare_routing(g, ref_route, wl.E)
    # a seeded sample, plus the tokens that end the shared expert's rows (its last tile) and the
    # largest and smallest routed segments (their tail tiles), from the oracle's own grouping
    p = oracle.permute(ref_route["ids"], wl.E)
    nz = np.nonzero(p["counts"])[0]
    big, small = nz[np.argmax(p["counts"][nz])], nz[np.argmin(p["counts"][nz])]
    ends = []
    for e in (big, small):
        last = p["offsets"][e + 1] - 1
        ends += [int(p["perm"][r]) for r in range(max(p["offsets"][e], last - 3), last + 1)]
    extra = [4095, 4094, 3840] + ends
    rows = sorted(set(sample_tokens(4096, 256, 5).tolist()) | set(extra))
    rows = np.array([t for t in rows if not diff[t]], dtype=np.int64)
    print(f"c5 output sample: {len(rows)} tokens; largest segment: expert {big} "
          f"({p['counts'][big]} rows), smallest: expert {small} ({p['counts'][small]} rows)")
    ref = oracle_pool.moe_forward(wl, x, wr, b, rows)
    compare_output(g["out"][rows], ref["out"])
    del torch
