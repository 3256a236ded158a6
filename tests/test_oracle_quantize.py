"""Pins of the oracle's group quantizer against what the definition fixes.

Definition ("Strata" MoE tuning notes, lpnh.cn/news/2730718, §2.1 group_quantize
sketch): per 128-wide group along the input dimension, scale = absmax / 7 and
q = clamp(round(w / scale), -8, 7). None of the checks below re-types the
oracle's formula: they use exact rational arithmetic and exhaustive search.
"""
import bisect
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import strata_oracle as so
from workloads import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quantize_cases.json")


# ---------------------------------------------------------------- exact references

def _all_fp16_positive():
    bits = np.arange(1, 0x7C00, dtype=np.uint16)          # every positive finite fp16
    vals = bits.view(np.float16)
    return [Fraction(float(v)) for v in vals], bits


_POS16, _POS16_BITS = _all_fp16_positive()


def nearest_fp16_exact(x: Fraction) -> Fraction:
    """Nearest fp16 to a non-negative rational by exhaustive table, ties to even bits."""
    if x == 0:
        return Fraction(0)
    i = bisect.bisect_left(_POS16, x)
    cands = []
    if i < len(_POS16):
        cands.append(i)
    if i > 0:
        cands.append(i - 1)
    else:
        cands.append(None)                                  # zero is the lower neighbour
    best = None
    for c in cands:
        v = Fraction(0) if c is None else _POS16[c]
        even = True if c is None else int(_POS16_BITS[c]) % 2 == 0
        d = abs(v - x)
        key = (d, not even)
        if best is None or key < best[0]:
            best = (key, v)
    return best[1]


def brute_quantize_group(ws, bits=4):
    """Exact: scale = fp16-nearest(absmax/qmax); q = argmin |w - q s| over the code range,
    ties even (qmax = 7, range [-8, 7] for 4 bits; 127 and [-128, 127] for 8)."""
    qmax = 2 ** (bits - 1) - 1
    fr = [Fraction(float(w)) for w in ws]
    a = max(abs(v) for v in fr)
    s = nearest_fp16_exact(a / qmax)
    qs = []
    for v in fr:
        if s == 0:
            qs.append(0)
            continue
        best = None
        for q in range(-qmax - 1, qmax + 1):
            key = (abs(v - q * s), q % 2)                    # prefer the even code on a tie
            if best is None or key < best[0]:
                best = (key, q)
        qs.append(best[1])
    return s, qs


def _groups_from(w16, n_groups, rng, group=128):
    rows = rng.integers(0, w16.shape[0], n_groups)
    gs = rng.integers(0, w16.shape[1] // group, n_groups)
    return [(int(r), int(g)) for r, g in zip(rows, gs)]


# ---------------------------------------------------------------- tests

def test_golden_hand_built_groups():
    cases = json.load(open(GOLDEN))
    for g in cases["groups"]:
        w = np.zeros((1, 128), dtype=np.float16)
        for i, v in g["nonzero"]:
            w[0, i] = v
        codes, scales = oracle.quantize_groups(w)
        assert float(scales[0, 0]) == g["scale"], g["why"]
        q = oracle.unpack_codes(codes)[0]
        expect = np.zeros(128, dtype=np.int8)
        for i, c in g["codes_nonzero"]:
            expect[i] = c
        np.testing.assert_array_equal(q, expect, err_msg=g["why"])


def test_golden_packing():
    cases = json.load(open(GOLDEN))["packing"]
    for (a, b), byte in cases["pairs"]:
        q = np.array([[a, b]], dtype=np.int8)
        assert int(oracle.pack_codes(q)[0, 0]) == byte
        np.testing.assert_array_equal(oracle.unpack_codes(np.array([[byte]], np.uint8))[0], [a, b])


@pytest.mark.parametrize("scale_exp", [0, -6, -14, -20])
def test_exact_brute_force_random_groups(scale_exp):
    """Random N(0,0.02) groups, also rescaled into fp16's subnormal range."""
    rng = np.random.default_rng(100 + scale_exp)
    w = gen.expert_weight(0, 0, 0, "gate", 16, 1024)
    w = (w.astype(np.float32) * np.float32(2.0 ** scale_exp)).astype(np.float16)
    codes, scales = oracle.quantize_groups(w)
    q = oracle.unpack_codes(codes)
    for r, g in _groups_from(w, 12, rng):
        s, qs = brute_quantize_group(w[r, g * 128:(g + 1) * 128])
        assert Fraction(float(scales[r, g])) == s
        np.testing.assert_array_equal(q[r, g * 128:(g + 1) * 128], qs)


def test_round_trip_bound_and_absmax():
    w = gen.expert_weight(0, 0, 1, "up", 64, 2048)
    codes, scales = oracle.quantize_groups(w)
    q = oracle.unpack_codes(codes).astype(np.int64)
    s = scales.astype(np.float64)
    wg = w.astype(np.float64).reshape(64, 16, 128)
    qg = q.reshape(64, 16, 128)
    # |w - q s| <= s/2 holds exactly: check with rationals on a sample, fp64 (exact here) on all
    err = np.abs(wg - qg * s[..., None])
    assert np.all(err <= s[..., None] / 2)
    for r, g in [(0, 0), (13, 7), (63, 15)]:
        sf = Fraction(float(s[r, g]))
        for i in range(128):
            assert abs(Fraction(float(wg[r, g, i])) - qg[r, g, i] * sf) <= sf / 2
    # the group's absmax element maps to +-7, and -8 never occurs
    am = np.abs(wg).argmax(axis=-1)
    top = np.take_along_axis(qg, am[..., None], axis=-1)[..., 0]
    topw = np.take_along_axis(wg, am[..., None], axis=-1)[..., 0]
    np.testing.assert_array_equal(np.abs(top), 7)
    np.testing.assert_array_equal(np.sign(top), np.sign(topw))
    assert q.min() >= -7


def test_idempotent():
    """Quantizing w = q0*s0 (exact in fp16, one +-7 per group) returns (q0, s0)."""
    rng = np.random.default_rng(11)
    n, kdim = 32, 1024
    q0 = rng.integers(-7, 8, (n, kdim)).astype(np.int8)
    q0[:, ::128] = rng.choice([-7, 7], (n, kdim // 128))
    # scales with <= 8 significant bits so that every q*s (q <= 7, 3 bits) is exact in fp16
    mant = rng.integers(128, 256, (n, kdim // 128))
    s0 = (mant * 2.0 ** rng.integers(-20, -8, (n, kdim // 128))).astype(np.float16)
    assert np.all(s0.astype(np.float64) == mant * 2.0 ** np.log2(s0.astype(np.float64) / mant))
    w64 = q0.reshape(n, -1, 128) * s0.astype(np.float64)[..., None]
    w = w64.reshape(n, kdim).astype(np.float16)
    assert np.array_equal(w.astype(np.float64), w64.reshape(n, kdim))
    codes, scales = oracle.quantize_groups(w)
    np.testing.assert_array_equal(scales, s0)
    np.testing.assert_array_equal(oracle.unpack_codes(codes), q0)


def test_dequantize_layout_by_hand():
    # 2 rows x 256: row 0 group 0 codes 1, group 1 codes -2; row 1 group 0 codes 7, group 1 codes -7
    q = np.zeros((2, 256), dtype=np.int8)
    q[0, :128], q[0, 128:] = 1, -2
    q[1, :128], q[1, 128:] = 7, -7
    sc = np.array([[0.5, 0.25], [2.0, 1.0]], dtype=np.float16)
    d = oracle.dequantize(oracle.pack_codes(q), sc)
    assert d[0, 0] == 0.5 and d[0, 200] == -0.5 and d[1, 5] == 14.0 and d[1, 255] == -7.0


def test_shape_and_finiteness_errors():
    with pytest.raises(ValueError):
        oracle.quantize_groups(np.zeros((2, 100), dtype=np.float16))
    bad = np.zeros((1, 128), dtype=np.float16)
    bad[0, 3] = np.inf
    with pytest.raises(ValueError):
        oracle.quantize_groups(bad)
    with pytest.raises(ValueError):
        oracle.quantize_groups(np.zeros((1, 128), dtype=np.float16), group=32)
    with pytest.raises(ValueError):
        oracle.quantize_groups(np.zeros((1, 128), dtype=np.float16), group=256)  # 128 % 256


# ---------------------------------------------------------------- other group sizes

@pytest.mark.parametrize("group", [64, 256])
def test_other_group_sizes_brute_force(group):
    """The group size is a parameter of the sketch: every group of G weights gets its own
    absmax / 7 scale; checked group by group by exact rational search."""
    rng = np.random.default_rng(7 + group)
    w = gen.expert_weight(0, 0, 2, "down", 8, 1024)
    codes, scales = oracle.quantize_groups(w, group=group)
    assert scales.shape == (8, 1024 // group) and codes.shape == (8, 512)
    q = oracle.unpack_codes(codes)
    for r, g in _groups_from(w, 8, rng, group):
        s, qs = brute_quantize_group(w[r, g * group:(g + 1) * group])
        assert Fraction(float(scales[r, g])) == s
        np.testing.assert_array_equal(q[r, g * group:(g + 1) * group], qs)


@pytest.mark.parametrize("group", [64, 256])
def test_other_group_sizes_round_trip_and_dequantize(group):
    w = gen.expert_weight(0, 0, 3, "gate", 16, 512)
    codes, scales = oracle.quantize_groups(w, group=group)
    d = oracle.dequantize(codes, scales)             # the group size follows from the shapes
    s = np.repeat(scales.astype(np.float64), group, axis=1)
    assert np.all(np.abs(w.astype(np.float64) - d) <= s / 2)
    # a 64-group split of the same row refines the 128-group scales: each 64-scale <= its 128-scale
    if group == 64:
        _, s128 = oracle.quantize_groups(w)
        assert np.all(scales.astype(np.float64).reshape(16, -1, 2).max(-1) == s128.astype(np.float64))


def test_dequantize_layout_by_hand_group_64():
    # 1 row x 128 in two 64-groups: codes 3 then -1, scales 0.5 and 4
    q = np.zeros((1, 128), dtype=np.int8)
    q[0, :64], q[0, 64:] = 3, -1
    sc = np.array([[0.5, 4.0]], dtype=np.float16)
    d = oracle.dequantize(oracle.pack_codes(q), sc)
    assert d[0, 0] == 1.5 and d[0, 63] == 1.5 and d[0, 64] == -4.0 and d[0, 127] == -4.0


def test_fp16_quotient_reading_differs_rarely():
    """The literal fp16 quotient reading: count where it differs from the exact one."""
    w = gen.expert_weight(0, 0, 3, "gate", 256, 4096)
    c_exact, s_exact = oracle.quantize_groups(w)
    c_f16, s_f16 = oracle.quantize_groups_f16_quotient(w)
    np.testing.assert_array_equal(s_exact, s_f16)
    diff = np.count_nonzero(oracle.unpack_codes(c_exact) != oracle.unpack_codes(c_f16))
    assert diff / w.size < 1e-3      # rare; reported, not a failure of either reading


def test_planted_rounding_mistake_is_caught(monkeypatch):
    """Round-half-away (a plausible slip) must fail the hand-built tie group."""
    monkeypatch.setattr(so.np, "rint", lambda a: np.trunc(a + np.copysign(0.5, a)))
    cases = json.load(open(GOLDEN))
    g = cases["groups"][0]
    w = np.zeros((1, 128), dtype=np.float16)
    for i, v in g["nonzero"]:
        w[0, i] = v
    q = so.unpack_codes(so.quantize_groups(w)[0])[0]
    expect = np.zeros(128, dtype=np.int8)
    for i, c in g["codes_nonzero"]:
        expect[i] = c
    assert not np.array_equal(q, expect)


# ---------------------------------------------------------------- 8-bit codes

def test_golden_hand_built_groups_8bit():
    cases = json.load(open(GOLDEN))
    for g in cases["groups_8bit"]:
        w = np.zeros((1, 128), dtype=np.float16)
        for i, v in g["nonzero"]:
            w[0, i] = v
        codes, scales = oracle.quantize_groups(w, bits=8)
        assert codes.dtype == np.int8 and codes.shape == (1, 128)
        assert float(scales[0, 0]) == g["scale"], g["why"]
        expect = np.zeros(128, dtype=np.int8)
        for i, c in g["codes_nonzero"]:
            expect[i] = c
        np.testing.assert_array_equal(codes[0], expect, err_msg=g["why"])


@pytest.mark.parametrize("scale_exp,group", [(0, 128), (-14, 128), (0, 64), (-6, 256)])
def test_exact_brute_force_random_groups_8bit(scale_exp, group):
    """8-bit codes: every sampled group equals the exact-rational search over [-128, 127]."""
    rng = np.random.default_rng(300 + scale_exp + group)
    w = gen.expert_weight(0, 0, 4, "up", 8, 1024)
    w = (w.astype(np.float32) * np.float32(2.0 ** scale_exp)).astype(np.float16)
    codes, scales = oracle.quantize_groups(w, group=group, bits=8)
    for r, g in _groups_from(w, 6, rng, group):
        s, qs = brute_quantize_group(w[r, g * group:(g + 1) * group], bits=8)
        assert Fraction(float(scales[r, g])) == s
        np.testing.assert_array_equal(codes[r, g * group:(g + 1) * group], qs)


def test_round_trip_bound_and_absmax_8bit():
    w = gen.expert_weight(0, 0, 5, "down", 32, 2048)
    codes, scales = oracle.quantize_groups(w, bits=8)
    q = codes.astype(np.int64).reshape(32, 16, 128)
    s = scales.astype(np.float64)
    wg = w.astype(np.float64).reshape(32, 16, 128)
    assert np.all(np.abs(wg - q * s[..., None]) <= s[..., None] / 2)
    am = np.abs(wg).argmax(axis=-1)
    top = np.take_along_axis(q, am[..., None], axis=-1)[..., 0]
    topw = np.take_along_axis(wg, am[..., None], axis=-1)[..., 0]
    np.testing.assert_array_equal(np.abs(top), 127)
    np.testing.assert_array_equal(np.sign(top), np.sign(topw))
    assert q.min() >= -127                  # -128 never occurs
    # 8-bit codes resolve the same weights ~18x finer than 4-bit ones (scale ratio 127 / 7)
    _, s4 = oracle.quantize_groups(w)
    ratio = s4.astype(np.float64) / s
    assert np.all(np.abs(ratio - 127 / 7) < 127 / 7 * 2e-3)


def test_idempotent_8bit():
    """Quantizing w = q0*s0 (exact in fp16, one +-127 per group) returns (q0, s0)."""
    rng = np.random.default_rng(12)
    n, kdim = 16, 512
    q0 = rng.integers(-127, 128, (n, kdim)).astype(np.int8)
    q0[:, ::128] = rng.choice([-127, 127], (n, kdim // 128))
    # scales with <= 4 significant bits: q*s (7 + 4 bits) is exact in fp16
    mant = rng.integers(8, 16, (n, kdim // 128))
    s0 = (mant * 2.0 ** rng.integers(-18, -10, (n, kdim // 128))).astype(np.float16)
    w64 = q0.reshape(n, -1, 128) * s0.astype(np.float64)[..., None]
    w = w64.reshape(n, kdim).astype(np.float16)
    assert np.array_equal(w.astype(np.float64), w64.reshape(n, kdim))
    codes, scales = oracle.quantize_groups(w, bits=8)
    np.testing.assert_array_equal(scales, s0)
    np.testing.assert_array_equal(codes, q0)


def test_dequantize_layout_by_hand_8bit():
    # int8 codes are one per byte, told apart from packed 4-bit codes by their dtype
    q = np.zeros((1, 256), dtype=np.int8)
    q[0, 0], q[0, 127], q[0, 128], q[0, 255] = -127, 3, 100, -1
    sc = np.array([[0.5, 0.25]], dtype=np.float16)
    d = oracle.dequantize(q, sc)
    assert d[0, 0] == -63.5 and d[0, 127] == 1.5 and d[0, 128] == 25.0 and d[0, 255] == -0.25
    assert d[0, 1] == 0.0


def test_bits_argument_errors():
    with pytest.raises(ValueError):
        oracle.quantize_groups(np.zeros((1, 128), dtype=np.float16), bits=2)
    with pytest.raises(ValueError):
        oracle.quantize_groups(np.zeros((1, 128), dtype=np.float16), bits=16)


def test_planted_divisor_mistake_is_caught_8bit(monkeypatch):
    """Dividing the absmax by 128 instead of 127 (a plausible slip) must fail the golden groups."""
    real = so.code_range
    monkeypatch.setattr(so, "code_range", lambda bits: (real(bits)[0], real(bits)[1], 128.0)
                        if bits == 8 else real(bits))
    g = json.load(open(GOLDEN))["groups_8bit"][0]
    w = np.zeros((1, 128), dtype=np.float16)
    for i, v in g["nonzero"]:
        w[0, i] = v
    codes, scales = so.quantize_groups(w, bits=8)
    assert float(scales[0, 0]) != g["scale"]


# ---------------------------------------------------------------- the fp16-quotient reading

def _fp16_rne(q):
    """Nearest fp16 to a positive rational (ties to an even significand), normal range only:
    written with Fractions, independent of numpy's float16 conversion."""
    from fractions import Fraction
    e = 0
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    while Fraction(2) ** e > q:
        e -= 1
    ulp = Fraction(2) ** (e - 10)
    m = q / ulp
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n * ulp


def _round_half_even(q):
    from fractions import Fraction
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n


def _disagreeing_pairs():
    """(absmax, w) fp16 pairs, as Fractions, whose exact quotient w/s is not a half-integer but
    rounds to one in fp16 (s = fp16(absmax / 7)), so that the two readings give different codes.
    Found by an exact search over 11-bit significands near the quotients 1.5, 2.5 and 3.5."""
    from fractions import Fraction
    found = []
    for target in (Fraction(3, 2), Fraction(5, 2), Fraction(7, 2)):
        done = False
        for S in range(1025, 2048):
            s = Fraction(S, 2 ** 13)
            for A in range(1024, 2048):        # absmax = A * 2^-11 must give this scale
                a = Fraction(A, 2 ** 11)
                if _fp16_rne(a / 7) != s or a < 7 * s * Fraction(99, 100):
                    continue
                for W in range(512, 2048):     # w = W * 2^-12 near target * s
                    w = Fraction(W, 2 ** 12)
                    if w > a:
                        break
                    q = w / s
                    if abs(q - target) > Fraction(1, 256) or q == target:
                        continue
                    if _round_half_even(q) != _round_half_even(_fp16_rne(q)):
                        found.append((a, w, q))
                        done = True
                        break
                if done:
                    break
            if done:
                break
    return found


def test_f16_quotient_reading_on_exact_rational_half_ties():
    """quantize_groups_f16_quotient (the literal fp16 reading: w/s rounded to fp16, then rounded
    half to even) against exact rational arithmetic, on groups built so that fp16(w/s) lands on a
    half-integer while w/s itself does not: the exact reading (quantize_groups) and the fp16
    reading must then give different codes, each the one the rational arithmetic predicts."""
    pairs = _disagreeing_pairs()
    assert len(pairs) == 3, pairs
    for a, w, q in pairs:
        g = np.zeros((1, 128), dtype=np.float16)
        g[0, 0] = float(a)
        g[0, 5] = float(w)
        g[0, 9] = -float(w)
        assert g[0, 0] == float(a) and g[0, 5] == float(w)   # exactly representable
        exact = so.unpack_codes(so.quantize_groups(g)[0])[0]
        lit = so.unpack_codes(so.quantize_groups_f16_quotient(g)[0])[0]
        q_exact, q_lit = _round_half_even(q), _round_half_even(_fp16_rne(q))
        assert q_exact != q_lit
        assert exact[5] == q_exact and exact[9] == -q_exact
        assert lit[5] == q_lit and lit[9] == -q_lit
        assert exact[0] == lit[0] == 7


def test_subnormal_scale_takes_the_clamp():
    """A group with absmax 10 * 2^-24 (a subnormal fp16) has absmax / 7 = 1.43 * 2^-24, which rounds
    to the scale 2^-24: the quotients are then the integers w / 2^-24 themselves, and the sketch's
    clamp to [-8, 7] decides the ends (+10 -> 7, -10 -> -8). With 8-bit codes (divisor 127) the
    scale 10/127 * 2^-24 rounds to 0 and every code is 0."""
    tiny = 2.0 ** -24
    vals = np.array([10, -10, 3, -3, 7, -8, 9, 0] * 16, dtype=np.float64) * tiny
    w = vals.astype(np.float16).reshape(1, 128)
    assert np.array_equal(w.astype(np.float64).ravel(), vals)        # exact in fp16
    codes, scales = oracle.quantize_groups(w)
    assert float(scales[0, 0]) == tiny
    q = oracle.unpack_codes(codes).astype(np.int64).ravel()
    expect = np.clip(np.array([10, -10, 3, -3, 7, -8, 9, 0] * 16), -8, 7)
    np.testing.assert_array_equal(q, expect)
    codes8, scales8 = oracle.quantize_groups(w, bits=8)
    assert float(scales8[0, 0]) == 0.0
    assert not np.asarray(codes8).any()
