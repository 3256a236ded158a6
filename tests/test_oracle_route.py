"""Pins of the oracle's router (softmax + top-k) and token permutation.

Router: "Strata" MoE tuning notes (lpnh.cn/news/2730718) §2.3, point 1 — top-k
selection and softmax fused; routing engine of the 102.7 tok/s write-up
(zwxr.cn/news/276292) §3.2 — softmax over the logits, partial sort for the top
k, ids out. Permutation: tokens routed to one expert are gathered into one
group of a grouped GEMM ("Strata" 3090 tuning, xdnf.cn/news/329730, §3.2).
"""
import math

import numpy as np
import pytest

import oracle
from oracle import strata_oracle as so
from workloads import gen


def brute_route(x_bits, wr, bias, k):
    """Pure-Python: fsum logits, exp softmax, repeated selection of the max (lowest id on ties)."""
    x = gen.bf16_bits_to_f32(x_bits).astype(np.float64)
    T, H = x.shape
    E = wr.shape[0]
    ids, gates = [], []
    for t in range(T):
        logit = []
        for e in range(E):
            s = math.fsum(float(x[t, h]) * float(wr[e, h]) for h in range(H))
            logit.append(s + (float(bias[e]) if bias is not None else 0.0))
        m = max(logit)
        ex = [math.exp(v - m) for v in logit]
        z = math.fsum(ex)
        p = [v / z for v in ex]
        left = list(range(E))
        row_i, row_g = [], []
        for _ in range(k):
            best = left[0]
            for e in left[1:]:
                if p[e] > p[best]:
                    best = e
            row_i.append(best)
            row_g.append(p[best])
            left.remove(best)
        ids.append(row_i)
        gates.append(row_g)
    return np.array(ids), np.array(gates)


@pytest.mark.parametrize("T,H,E,k,with_bias", [(5, 128, 6, 2, False), (4, 256, 9, 3, True),
                                               (3, 128, 4, 4, True), (6, 128, 5, 1, False)])
def test_route_brute_force(T, H, E, k, with_bias):
    rng = np.random.default_rng(T * 100 + E)
    x = gen.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = (rng.standard_normal((E, H)) * 0.05).astype(np.float32)
    b = (rng.standard_normal(E) * 0.3).astype(np.float32) if with_bias else None
    r = oracle.route_topk(x, wr, b, k)
    bi, bg = brute_route(x, wr, b, k)
    np.testing.assert_array_equal(r["ids"], bi)
    np.testing.assert_allclose(r["gates"], bg, rtol=1e-12, atol=0)


def test_full_sort_and_normalisation():
    rng = np.random.default_rng(3)
    x = gen.f32_to_bf16_bits(rng.standard_normal((64, 512)).astype(np.float32))
    wr = (rng.standard_normal((40, 512)) * 0.02).astype(np.float32)
    r = oracle.route_topk(x, wr, None, 40)
    np.testing.assert_allclose(r["probs"].sum(axis=1), 1.0, rtol=0, atol=1e-14)
    for t in range(64):
        order = sorted(range(40), key=lambda e: (-r["probs"][t, e], e))
        assert list(r["ids"][t]) == order                            # k = E: every id, sorted
    r5 = oracle.route_topk(x, wr, None, 5)
    np.testing.assert_array_equal(r5["ids"], r["ids"][:, :5])        # top-k is a prefix of the sort


def test_zero_router_is_uniform_with_lowest_ids():
    x = gen.activations(7, 256, 0)
    wr = np.zeros((12, 256), dtype=np.float32)
    r = oracle.route_topk(x, wr, None, 3)
    np.testing.assert_allclose(r["probs"], 1 / 12, rtol=1e-15)
    np.testing.assert_array_equal(r["ids"], np.tile([0, 1, 2], (7, 1)))    # ties -> lower id
    assert np.all(r["gap"] == 0)


def test_bias_shift_invariance_and_renorm():
    rng = np.random.default_rng(5)
    x = gen.f32_to_bf16_bits(rng.standard_normal((16, 256)).astype(np.float32))
    wr = (rng.standard_normal((10, 256)) * 0.05).astype(np.float32)
    b = (rng.standard_normal(10)).astype(np.float32)
    r1 = oracle.route_topk(x, wr, b, 3)
    r2 = oracle.route_topk(x, wr, (b + np.float32(4.0)).astype(np.float32), 3)
    np.testing.assert_array_equal(r1["ids"], r2["ids"])
    np.testing.assert_allclose(r1["gates"], r2["gates"], rtol=1e-6)
    rn = oracle.route_topk(x, wr, b, 3, renorm=True)
    np.testing.assert_allclose(rn["gates"].sum(axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(rn["gates"] * r1["gates"].sum(axis=1, keepdims=True), r1["gates"], rtol=1e-14)


def brute_permute(ids, E):
    T, k = ids.shape
    pairs = sorted((int(ids[t, j]), t, j) for t in range(T) for j in range(k))
    perm = [t for (_, t, _) in pairs]
    inv = np.zeros((T, k), dtype=np.int64)
    for r, (_, t, j) in enumerate(pairs):
        inv[t, j] = r
    counts = [sum(1 for p in pairs if p[0] == e) for e in range(E)]
    return counts, perm, inv


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (13, 7, 3), (32, 16, 16), (50, 300, 8), (0, 5, 2)])
def test_permute_brute_force(T, E, k):
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), np.int32)
    p = oracle.permute(ids, E)
    counts, perm, inv = brute_permute(ids, E)
    np.testing.assert_array_equal(p["counts"], counts)
    np.testing.assert_array_equal(p["perm"], perm)
    np.testing.assert_array_equal(p["inv"], inv)
    assert p["counts"].sum() == T * k and p["offsets"][-1] == T * k
    np.testing.assert_array_equal(np.diff(p["offsets"]), p["counts"])
    if T:
        # perm and inv are inverse bijections: the row of (t, j) holds token t
        np.testing.assert_array_equal(p["perm"][p["inv"]], np.repeat(np.arange(T)[:, None], k, 1))
        assert sorted(p["inv"].reshape(-1).tolist()) == list(range(T * k))


def test_all_tokens_to_one_expert():
    ids = np.zeros((9, 1), dtype=np.int32) + 3
    p = oracle.permute(ids, 5)
    np.testing.assert_array_equal(p["counts"], [0, 0, 0, 9, 0])
    np.testing.assert_array_equal(p["perm"], np.arange(9))


def test_planted_tie_break_mistake_is_caught(monkeypatch):
    """Taking the last of equal probabilities (a plausible slip) must fail the zero-router pin."""
    real = np.argsort

    def backwards(a, axis=-1, kind=None):
        a = np.asarray(a)
        n = a.shape[axis]
        flipped = np.flip(a, axis=axis)
        return n - 1 - real(flipped, axis=axis, kind="stable")    # ascending, ties -> higher id
    monkeypatch.setattr(so.np, "argsort", backwards)
    x = gen.activations(2, 128, 0)
    r = so.route_topk(x, np.zeros((6, 128), np.float32), None, 2)
    assert not np.array_equal(r["ids"], np.tile([0, 1], (2, 1)))


def test_dot_l2_is_the_norm_of_each_logits_product_terms():
    """route_topk's dot_l2[t, e] = sqrt(sum_h (x[t,h] * w[e,h])^2), by pure-Python loops."""
    rng = np.random.default_rng(4)
    x = gen.f32_to_bf16_bits(rng.standard_normal((3, 16)).astype(np.float32))
    w = (rng.standard_normal((5, 16)) * 0.3).astype(np.float32)
    r = oracle.route_topk(x, w, None, 2)
    xf = oracle.bf16_to_f64(x)
    for t in range(3):
        for e in range(5):
            s = 0.0
            for h in range(16):
                s += (float(xf[t, h]) * float(w[e, h])) ** 2
            assert abs(r["dot_l2"][t, e] - math.sqrt(s)) <= 1e-12 * math.sqrt(s)
