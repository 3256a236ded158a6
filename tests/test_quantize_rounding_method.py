"""The rounding method the group-quantize kernel uses, checked on the CPU.

The kernel never divides per weight. It rounds w * RN32(1/s) to an integer q, computes the
residual w - q*s (exact in fp32) and, where that residual is exactly +-s/2, moves q to its even
neighbour. The claim is that this equals round-half-even of the exact quotient w / s, which is
what the oracle takes ("Strata" MoE tuning notes, lpnh.cn/news/2730718, §2.1: round(w / scale),
torch's round being half to even), for every pair of fp16 values a group can hold. Here the
method's fp32 steps are emulated with numpy float32, and the reference is the oracle's own
quantizer on groups built to contain the pairs. Nothing here runs on or imports the library.
"""
import numpy as np

from oracle import strata_oracle as so


def _method(w: np.ndarray, s: float) -> np.ndarray:
    """q from the kernel's steps, emulated in fp32 (the residual is exact, so fp64 holds it)."""
    inv = np.float32(1.0) / np.float32(s)
    q = np.rint((w.astype(np.float32) * inv).astype(np.float32)).astype(np.float64)
    r = w - q * s
    odd = (q.astype(np.int64) & 1) != 0
    return q + ((r == 0.5 * s) & odd) - ((r == -0.5 * s) & odd)


def _exact_rne(w: np.ndarray, s: float) -> np.ndarray:
    """Round half to even of w / s, decided with the fp64 quotient of two fp16 values."""
    x = w / s
    fl = np.floor(x)
    fr = x - fl
    return np.where(fr > 0.5, fl + 1, np.where(fr < 0.5, fl, fl + (fl % 2 != 0)))


def test_method_equals_exact_round_half_even_for_every_fp16_weight():
    w_all = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    w_all = np.concatenate([w_all, -w_all[1:]])
    rng = np.random.default_rng(7)
    scales = np.concatenate([np.arange(1, 0x7C00, 251, dtype=np.uint16),
                             rng.integers(1, 0x7C00, 60).astype(np.uint16)])
    ties = 0
    for qmax in (7, 127):
        for sb in scales:
            s = float(np.uint16(sb).view(np.float16))
            w = w_all[np.abs(w_all) <= s * qmax * (1 + 2.0 ** -11)]
            if w.size == 0:
                continue
            got = _method(w, s)
            want = _exact_rne(w, s)
            assert np.array_equal(got, want), (s, w[got != want][:4])
            r = w - np.rint(w / s) * s
            assert np.all(r.astype(np.float32) == r)  # the residual needs no rounding in fp32
            ties += int(np.sum(np.abs(w / s - np.floor(w / s)) == 0.5))
    assert ties > 1000  # the sample holds many exact ties, both signs


def test_method_matches_the_oracle_on_tie_groups():
    # groups whose absmax fixes s = absmax / 7 exactly and whose other weights sit on half-steps
    for absmax in (7.0, 0.875, 7.0 * 2.0 ** -12, 3.5):
        s = absmax / 7.0
        half_steps = np.arange(-14, 15) * 0.5 * s            # every half-step of s in [-7s, 7s]
        w = np.concatenate([[absmax], half_steps, np.zeros(128 - 1 - half_steps.size)])
        w16 = w.astype(np.float16)
        assert np.array_equal(w16.astype(np.float64), w)     # all exactly representable
        codes, scales = so.quantize_groups(w16.reshape(1, 128))
        assert float(scales[0, 0]) == s
        q_oracle = so.unpack_codes(codes)[0].astype(np.float64)
        q_method = np.clip(_method(w, s), -8, 7)
        assert np.array_equal(q_method, q_oracle)
