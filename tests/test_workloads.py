"""The seeded workloads: determinism, distributions, and the stored Zipf strengths."""
import math

import numpy as np
import pytest

import oracle
from workloads import CONFIGS, ZIPF_ALPHA, gen


def test_generators_are_deterministic_and_per_tensor():
    wl = CONFIGS["c1"]
    a = gen.expert_weights(wl, 3)
    b = gen.expert_weights(wl, 3)
    for m1, m2 in zip(a, b):
        np.testing.assert_array_equal(m1, m2)
    assert a[0].shape == (wl.I, wl.H) and a[2].shape == (wl.H, wl.I)
    assert a[0].dtype == np.float16
    c = gen.expert_weights(wl, 4)
    assert not np.array_equal(a[0], c[0])
    np.testing.assert_array_equal(gen.activations(5, 64, 0), gen.activations(5, 64, 0))


def test_distributions():
    w = gen.expert_weight(0, 0, 0, "gate", 512, 1024).astype(np.float64)
    assert abs(w.std() - 0.02) < 5e-4 and abs(w.mean()) < 5e-4
    x = gen.bf16_bits_to_f32(gen.activations(256, 1024, 0)).astype(np.float64)
    assert abs(x.std() - 1.0) < 0.01


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5], dtype=np.float32)
    bits = gen.f32_to_bf16_bits(vals)
    back = gen.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa -> 1.0; 1 + 3*2^-8 -> 1 + 2^-6
    np.testing.assert_array_equal(back, [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5])


@pytest.mark.parametrize("key,layer", sorted(ZIPF_ALPHA))
def test_zipf_alpha_gives_80_percent(key, layer):
    wl = CONFIGS[key]
    x = gen.calibration_tokens(wl)
    b = gen.zipf_bias(wl.E, wl.seed, layer, ZIPF_ALPHA[(key, layer)])
    ids = oracle.route_topk(x, gen.router_weight(wl, layer), b, wl.k)["ids"]
    counts = np.sort(np.bincount(ids.reshape(-1), minlength=wl.E))[::-1]
    share = counts[:math.ceil(0.2 * wl.E)].sum() / counts.sum()
    assert 0.79 <= share <= 0.81
