"""Pins of the oracle's expert FFN and whole MoE layer.

Expert form: Gate/Up + Down projections ("GLM-5.3-Flash on one 4090",
haowenji.com/articles/x-2109226022155796480, §01) with a SiLU gate; top-k
weighted combine plus an always-on shared expert with gate 1 (same page, §01:
8 routed + 1 shared per token). Checks: pure-Python loops on tiny shapes (with
H != I so a transposed operand fails), dense equivalence against torch's own
SiLU when k = E and the router is zero, E = k = 1, token independence.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import strata_oracle as so
from workloads import gen


def make_layer(rng, E, H, I, shared, std=0.05, bits=4):
    ws = []
    for _ in range(E + shared):
        g = (rng.standard_normal((I, H)) * std).astype(np.float16)
        u = (rng.standard_normal((I, H)) * std).astype(np.float16)
        d = (rng.standard_normal((H, I)) * std).astype(np.float16)
        ws.append(tuple(oracle.quantize_groups(m, bits=bits) for m in (g, u, d)))
    return ws


def brute_ffn(x_row, wg, wu, wd):
    """Pure-Python loops, floats; w* are nested lists of dequantised values."""
    I, H = len(wg), len(wg[0])
    h = []
    for i in range(I):
        u = math.fsum(x_row[c] * wg[i][c] for c in range(H))
        v = math.fsum(x_row[c] * wu[i][c] for c in range(H))
        h.append(u / (1.0 + math.exp(-u)) * v)
    return [math.fsum(h[i] * wd[o][i] for i in range(I)) for o in range(len(wd))]


@pytest.mark.parametrize("T,E,k,shared,renorm", [(3, 3, 2, 0, False), (2, 4, 1, 1, False),
                                                  (4, 2, 2, 1, True)])
def test_layer_brute_force(T, E, k, shared, renorm):
    H, I = 256, 128
    rng = np.random.default_rng(T * 10 + E)
    ws = make_layer(rng, E, H, I, shared)
    x = gen.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = (rng.standard_normal((E, H)) * 0.05).astype(np.float32)
    res = oracle.moe_forward(x, wr, None, k, lambda e: ws[e], E, shared, renorm=renorm)
    ids, gates = res["route"]["ids"], res["route"]["gates"]
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    deq = [[oracle.dequantize(c, s).tolist() for (c, s) in w] for w in ws]
    for t in range(T):
        row = xf[t].tolist()
        acc = [0.0] * H
        for j in range(k):
            y = brute_ffn(row, *deq[ids[t, j]])
            acc = [a + gates[t, j] * b for a, b in zip(acc, y)]
        if shared:
            y = brute_ffn(row, *deq[E])
            acc = [a + b for a, b in zip(acc, y)]
        np.testing.assert_allclose(res["out"][t], acc, rtol=1e-10, atol=1e-12)


def torch_swiglu(x, wg, wu, wd):
    xt = torch.from_numpy(x)
    return (torch.nn.functional.silu(xt @ torch.from_numpy(wg).T) * (xt @ torch.from_numpy(wu).T)
            @ torch.from_numpy(wd).T).numpy()


def test_dense_equivalence_k_equals_e():
    """k = E, Wr = b = 0: every gate is 1/E and out = mean over experts of a dense SwiGLU."""
    E, H, I, T = 5, 384, 256, 6
    rng = np.random.default_rng(42)
    ws = make_layer(rng, E, H, I, 1)
    x = gen.activations(T, H, 1)
    res = oracle.moe_forward(x, np.zeros((E, H), np.float32), None, E, lambda e: ws[e], E, 1)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    dense = sum(torch_swiglu(xf, *[oracle.dequantize(c, s) for (c, s) in ws[e]]) for e in range(E)) / E
    dense += torch_swiglu(xf, *[oracle.dequantize(c, s) for (c, s) in ws[E]])
    np.testing.assert_allclose(res["out"], dense, rtol=1e-10, atol=1e-12)


def test_single_expert_is_one_ffn():
    H, I, T = 256, 384, 5
    rng = np.random.default_rng(9)
    ws = make_layer(rng, 1, H, I, 0)
    x = gen.activations(T, H, 2)
    wr = (rng.standard_normal((1, H)) * 0.02).astype(np.float32)
    res = oracle.moe_forward(x, wr, None, 1, lambda e: ws[e], 1, 0)
    np.testing.assert_array_equal(res["route"]["gates"], 1.0)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    ref = torch_swiglu(xf, *[oracle.dequantize(c, s) for (c, s) in ws[0]])
    np.testing.assert_allclose(res["out"], ref, rtol=1e-10, atol=1e-12)


def test_single_expert_is_one_ffn_8bit():
    """8-bit experts: E = k = 1 is one SwiGLU FFN of the dequantized weights, and those weights are
    within half a (127x finer) step of the fp16 ones."""
    H, I, T = 256, 128, 4
    rng = np.random.default_rng(19)
    ws = make_layer(rng, 1, H, I, 0, bits=8)
    assert all(c.dtype == np.int8 and c.shape[1] == s.shape[1] * 128 for (c, s) in ws[0])
    x = gen.activations(T, H, 6)
    wr = (rng.standard_normal((1, H)) * 0.02).astype(np.float32)
    res = oracle.moe_forward(x, wr, None, 1, lambda e: ws[e], 1, 0)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    ref = torch_swiglu(xf, *[oracle.dequantize(c, s) for (c, s) in ws[0]])
    np.testing.assert_allclose(res["out"], ref, rtol=1e-10, atol=1e-12)


def test_token_independence_and_residual():
    E, H, I, T, k = 6, 256, 128, 12, 2
    rng = np.random.default_rng(4)
    ws = make_layer(rng, E, H, I, 1)
    x = gen.activations(T, H, 3)
    wr = (rng.standard_normal((E, H)) * 0.05).astype(np.float32)
    full = oracle.moe_forward(x, wr, None, k, lambda e: ws[e], E, 1)["out"]
    sub = oracle.moe_forward(x, wr, None, k, lambda e: ws[e], E, 1, tokens=[7, 2, 11])["out"]
    np.testing.assert_allclose(sub, full[[7, 2, 11]], rtol=1e-12, atol=1e-15)   # BLAS blocking only
    res = oracle.moe_forward(x, wr, None, k, lambda e: ws[e], E, 1, residual=True)["out"]
    np.testing.assert_allclose(res - full, gen.bf16_bits_to_f32(x), rtol=0, atol=1e-12)


def test_planted_silu_sign_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(so, "silu", lambda u: u / (1.0 + np.exp(u)))
    E, H, I, T = 1, 256, 128, 2
    rng = np.random.default_rng(1)
    ws = make_layer(rng, E, H, I, 0)
    x = gen.activations(T, H, 5)
    res = so.moe_forward(x, np.zeros((1, H), np.float32), None, 1, lambda e: ws[e], 1, 0)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    ref = torch_swiglu(xf, *[oracle.dequantize(c, s) for (c, s) in ws[0]])
    assert not np.allclose(res["out"], ref, rtol=1e-6)


def test_expert_outputs_from_worker_processes_match_the_serial_oracle():
    """tests/oracle_pool.py evaluates the experts in spawned workers and hands them to
    oracle.moe_forward; the result must be the serial oracle's, bit for bit."""
    from helpers import OracleExperts
    import oracle_pool
    from workloads import CONFIGS
    wl = CONFIGS["c1"]
    x = gen.activations(9, wl.H, 3, name="pool")
    wr, b = gen.router_weight(wl), gen.router_bias(wl)
    tokens = [0, 2, 5, 8]
    ref = oracle.moe_forward(x, wr, b, wl.k, OracleExperts(wl), wl.E, wl.shared, tokens=tokens)
    got = oracle_pool.moe_forward(wl, x, wr, b, tokens, procs=2)
    np.testing.assert_array_equal(got["out"], ref["out"])


def test_bf16_half_ulp_of_the_output_comparison():
    """The allowance compare_output grants for the output's final bf16 rounding: half the spacing
    of bf16 values at the element (8 significant bits)."""
    from helpers import bf16_half_ulp
    v = np.array([1.0, 1.5, 8.0, 15.9, -8.22, 0.0, 2.0 ** -20])
    np.testing.assert_array_equal(bf16_half_ulp(v),
                                  [2.0 ** -8, 2.0 ** -8, 2.0 ** -5, 2.0 ** -5, 2.0 ** -5, 0.0,
                                   2.0 ** -28])
