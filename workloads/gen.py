"""Seeded input generators (no arithmetic of the MoE method lives here).

Every tensor has its own substream, `SeedSequence([seed, crc32(name)])`, so any
one expert of any layer can be regenerated alone (the oracle regenerates only
the experts a sampled token touches). Floats are drawn in fp32 and rounded to
nearest-even into their storage type: bf16 for activations, fp16 for expert
weights; router weights stay fp32.

Distributions (the five workload descriptions): activations N(0,1); expert
weights N(0,0.02); router weights N(0,0.02); optional Zipf(s) router bias
`alpha * ln p_rank(e)`, `p_r ~ r^-s` over a seeded permutation of the experts.
"""
from __future__ import annotations

import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import ZIPF_ALPHA, ZIPF_S, Workload

GATE, UP, DOWN = "gate", "up", "down"


def substream(seed: int, name: str) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), zlib.crc32(name.encode())]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even) and return the raw uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(T: int, H: int, seed: int = 0, name: str = "x") -> np.ndarray:
    """bf16 bits [T, H], values N(0,1)."""
    z = substream(seed, f"act/{name}/{T}x{H}").standard_normal((T, H), dtype=np.float32)
    return f32_to_bf16_bits(z)


def expert_weight(seed: int, layer: int, e: int, which: str, rows: int, cols: int,
                  std: float = 0.02) -> np.ndarray:
    """fp16 [rows, cols], values N(0, std), rounded to nearest-even."""
    z = substream(seed, f"w/{layer}/{e}/{which}").standard_normal((rows, cols), dtype=np.float32)
    z *= np.float32(std)
    return z.astype(np.float16)


def expert_weights(wl: Workload, e: int, layer: int = 0):
    """(gate [I,H], up [I,H], down [H,I]) fp16 of expert e (e == E is the shared one)."""
    s = wl.seed
    return (expert_weight(s, layer, e, GATE, wl.I, wl.H),
            expert_weight(s, layer, e, UP, wl.I, wl.H),
            expert_weight(s, layer, e, DOWN, wl.H, wl.I))


def expert_weights_many(wl: Workload, experts, layer: int = 0, threads: int = 0):
    """Generate several experts in parallel threads (numpy's generators release the GIL)."""
    experts = list(experts)
    if threads <= 0:
        import os
        threads = max(1, min(16, os.cpu_count() or 1))
    with ThreadPoolExecutor(threads) as ex:
        return list(ex.map(lambda e: expert_weights(wl, e, layer), experts))


def router_weight(wl: Workload, layer: int = 0) -> np.ndarray:
    """fp32 [E, H], N(0, 0.02)."""
    z = substream(wl.seed, f"router/{layer}").standard_normal((wl.E, wl.H), dtype=np.float32)
    return (z * np.float32(0.02)).astype(np.float32)


def zipf_bias(E: int, seed: int, layer: int, alpha: float, s: float = ZIPF_S) -> np.ndarray:
    """fp32 [E]: alpha * ln p_rank(e), p_r = r^-s / sum, ranks a seeded permutation."""
    rank = substream(seed, f"zipf_rank/{layer}").permutation(E)     # expert e has rank rank[e]+1
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** (-s)
    p /= p.sum()
    return (alpha * np.log(p[rank])).astype(np.float32)


def router_bias(wl: Workload, layer: int = 0, kind: str | None = None):
    """Router bias for the workload (None for the uniform router)."""
    kind = kind or wl.router
    if kind == "uniform":
        return None
    alpha = ZIPF_ALPHA.get((wl.key, layer))
    if alpha is None:
        raise KeyError(f"no calibrated Zipf alpha for {(wl.key, layer)}")
    return zipf_bias(wl.E, wl.seed, layer, alpha)


def calibration_tokens(wl: Workload, n: int = 2048) -> np.ndarray:
    return activations(n, wl.H, wl.seed, name=f"calib/{wl.key}")
