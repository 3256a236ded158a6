"""K1 group-quantize kernel vs the oracle: codes and scales bit-exact.

Definition: "Strata" MoE tuning notes (lpnh.cn/news/2730718), §2.1 group_quantize sketch.
"""
import json
import os

import numpy as np
import pytest

import oracle
from workloads import CONFIGS, gen

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quantize_cases.json")


def gpu_quantize(w16: np.ndarray, status=None, group=128, bits=4):
    import torch
    import int4_grouped_expert_gb300 as st
    n, k = w16.shape
    w = torch.from_numpy(w16).cuda()
    codes = torch.full((n, k * bits // 8), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((n, k // group), 7.0, dtype=torch.float16, device="cuda")
    if bits == 4:
        st.check(st.strata_quantize_groups(w, n, k, codes, scales, status, group_size=group),
                 "quantize")
    else:
        st.check(st.strata_quantize_groups_bits(w, n, k, codes, scales, status, group_size=group,
                                                bits=bits), "quantize")
    torch.cuda.synchronize()
    c = codes.cpu().numpy()
    return (c if bits == 4 else c.view(np.int8)), scales.cpu().numpy()


def assert_same(w16, group=128, bits=4):
    c, s = gpu_quantize(w16, group=group, bits=bits)
    rc, rs = oracle.quantize_groups(w16, group=group, bits=bits)
    np.testing.assert_array_equal(s.view(np.uint16), rs.view(np.uint16))
    np.testing.assert_array_equal(c, rc)


def test_golden_groups():
    cases = json.load(open(GOLDEN))["groups"]
    w = np.zeros((len(cases), 128), dtype=np.float16)
    for r, g in enumerate(cases):
        for i, v in g["nonzero"]:
            w[r, i] = v
    c, s = gpu_quantize(w)
    for r, g in enumerate(cases):
        assert float(s[r, 0]) == g["scale"], g["why"]
        expect = np.zeros(128, dtype=np.int8)
        for i, v in g["codes_nonzero"]:
            expect[i] = v
        np.testing.assert_array_equal(oracle.unpack_codes(c[r:r + 1])[0], expect, err_msg=g["why"])


@pytest.mark.parametrize("n,k", [(1, 128), (3, 256), (37, 1152), (129, 384), (1, 7168)])
def test_random_shapes(n, k):
    assert_same(gen.expert_weight(0, 0, n, "gate", n, k))


@pytest.mark.parametrize("scale_exp", [-10, -16, -22, 4])
def test_extreme_scales(scale_exp):
    w = gen.expert_weight(1, 0, 0, "up", 64, 512).astype(np.float32) * np.float32(2.0 ** scale_exp)
    assert_same(w.astype(np.float16))


def test_zero_groups_and_ties():
    rng = np.random.default_rng(0)
    w = np.zeros((8, 512), dtype=np.float16)
    w[1] = rng.integers(-7, 8, 512) * 0.5                 # exact multiples of half the scale
    w[2, :128] = np.arange(128) % 15 - 7.5                 # absmax 7.5: scale fp16(15/14)
    w[3] = np.where(rng.random(512) < 0.5, 6.5, -6.5)
    w[3, ::128] = 7.0
    assert_same(w)


@pytest.mark.parametrize("key", ["c2", "c5"])
def test_full_expert_matrices(key):
    wl = CONFIGS[key]
    for m in gen.expert_weights(wl, 5):
        assert_same(m)


def test_nonfinite_sets_status_and_marks_group():
    import torch
    import int4_grouped_expert_gb300 as st
    w = gen.expert_weight(0, 0, 9, "down", 4, 384)
    w[2, 130] = np.inf
    w[3, 5] = np.nan
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    c, s = gpu_quantize(w, status)
    rc, rs = oracle.quantize_groups(np.where(np.isfinite(w), w, 0).astype(np.float16))
    bad = {(2, 1), (3, 0)}
    for r in range(4):
        for g in range(3):
            if (r, g) in bad:
                assert np.isnan(s[r, g])
                assert not c[r, g * 64:(g + 1) * 64].any()
            else:
                assert s[r, g] == rs[r, g]
                np.testing.assert_array_equal(c[r, g * 64:(g + 1) * 64], rc[r, g * 64:(g + 1) * 64])
    rc_, v = st.strata_read_status(status)
    assert rc_ == st.STATUS_NAMES.index("STRATA_ERR_DEVICE_STATUS") and v & st.STRATA_DEV_NONFINITE
    rc_, v = st.strata_read_status(status)                 # read clears the word
    assert rc_ == 0 and v == 0


def test_argument_errors_on_device_pointers():
    import torch
    import int4_grouped_expert_gb300 as st
    w = torch.zeros(4, 256, dtype=torch.float16, device="cuda")
    c = torch.zeros(4, 128, dtype=torch.uint8, device="cuda")
    s = torch.zeros(4, 2, dtype=torch.float16, device="cuda")
    assert st.strata_quantize_groups(w, 4, 200, c, s) == 2                     # SHAPE
    assert st.strata_quantize_groups(w, 4, 256, c, s, group_size=32) == 3      # UNSUPPORTED
    assert st.strata_quantize_groups(w.view(-1)[1:].data_ptr(), 1, 128, c, s) == 1  # misaligned
    assert st.strata_quantize_groups(w, 0, 256, c, s) == 0                     # empty


@pytest.mark.parametrize("group", [64, 256])
@pytest.mark.parametrize("n,k", [(1, 256), (37, 1280), (5, 7168)])
def test_other_group_sizes(group, n, k):
    """Group sizes 64 and 256: codes and scales bit-exact against the oracle."""
    w = gen.expert_weight(2, 0, n, "down", n, k).astype(np.float32)
    w *= np.float32(2.0 ** (-6 if group == 64 else 2))
    assert_same(w.astype(np.float16), group=group)


# ---------------------------------------------------------------- 8-bit codes

def test_golden_groups_8bit():
    for g in json.load(open(GOLDEN))["groups_8bit"]:
        w = np.zeros((1, 128), dtype=np.float16)
        for i, v in g["nonzero"]:
            w[0, i] = v
        c, s = gpu_quantize(w, bits=8)
        assert float(s[0, 0]) == g["scale"], g["why"]
        expect = np.zeros(128, dtype=np.int8)
        for i, q in g["codes_nonzero"]:
            expect[i] = q
        np.testing.assert_array_equal(c[0], expect, err_msg=g["why"])


@pytest.mark.parametrize("group", [64, 128, 256])
@pytest.mark.parametrize("n,k", [(1, 256), (37, 1280), (5, 7168)])
def test_8bit_codes_match_oracle(group, n, k):
    """8-bit codes: scale = absmax / 127, one int8 code per byte; bit-exact against the oracle."""
    w = gen.expert_weight(3, 0, n, "gate", n, k)
    assert_same(w, group=group, bits=8)


@pytest.mark.parametrize("scale_exp", [-20, -14, 0, 8])
def test_8bit_extreme_scales(scale_exp):
    w = gen.expert_weight(4, 0, 1, "up", 16, 1024).astype(np.float32)
    w = (w * np.float32(2.0 ** scale_exp)).astype(np.float16)
    assert_same(w, bits=8)


def test_8bit_zero_groups_and_argument_errors():
    import torch
    import int4_grouped_expert_gb300 as st
    w16 = np.zeros((3, 384), dtype=np.float16)
    w16[1, 128:256] = np.float16(0.25)
    assert_same(w16, bits=8)
    w = torch.zeros(4, 256, dtype=torch.float16, device="cuda")
    c = torch.zeros(4, 256, dtype=torch.uint8, device="cuda")
    s = torch.zeros(4, 2, dtype=torch.float16, device="cuda")
    assert st.strata_quantize_groups_bits(w, 4, 256, c, s, bits=2) == 3          # UNSUPPORTED
    assert st.strata_quantize_groups_bits(w, 4, 200, c, s, bits=8) == 2          # SHAPE
    assert st.strata_quantize_groups_bits(w, 0, 256, c, s, bits=8) == 0          # empty


@pytest.mark.parametrize("group", [64, 128, 256])
def test_subnormal_scales_take_the_clamp(group):
    """Groups whose absmax is a few subnormal steps (2^-24): the scale rounds coarsely to a
    subnormal fp16 and the clamp to [-8, 7] decides the ends (the kernel's exact-quotient branch
    for scales below the smallest normal fp16), beside ordinary groups in the same rows."""
    rng = np.random.default_rng(group)
    n, k = 6, 4 * group
    steps = rng.integers(-12, 13, (n, k)).astype(np.float64)
    w = (steps * 2.0 ** -24).astype(np.float16)
    w[:, group:2 * group] = (rng.standard_normal((n, group)) * 0.02).astype(np.float16)
    for bits in (4, 8):
        assert_same(w, group=group, bits=bits)
