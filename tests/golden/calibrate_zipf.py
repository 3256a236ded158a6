"""Find the Zipf router-bias strength alpha for each skewed workload layer.

Bisects alpha so that, on a separate seeded 2048-token calibration batch routed
by the oracle, the 20% most-used experts take 80% of the routes (the pages'
hot-expert statistic: "Strata" 3090 tuning, xdnf.cn/news/329730, §2.1). Prints
the table that workloads/configs.py stores; tests/test_workloads.py re-checks
each stored value.

    python tests/golden/calibrate_zipf.py
"""
from __future__ import annotations

import math
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))

from oracle import route_topk  # noqa: E402
from workloads import CONFIGS, gen  # noqa: E402


def top20_share(wl, layer, alpha, x, wr):
    b = gen.zipf_bias(wl.E, wl.seed, layer, alpha)
    ids = route_topk(x, wr, b, wl.k)["ids"]
    counts = np.sort(np.bincount(ids.reshape(-1), minlength=wl.E))[::-1]
    top = math.ceil(0.2 * wl.E)
    return counts[:top].sum() / counts.sum()


def calibrate(wl, layer, target=0.80):
    x = gen.calibration_tokens(wl)
    wr = gen.router_weight(wl, layer)
    lo, hi = 0.0, 2.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if top20_share(wl, layer, mid, x, wr) < target:
            lo = mid
        else:
            hi = mid
    alpha = round(hi, 6)
    return alpha, top20_share(wl, layer, alpha, x, wr)


if __name__ == "__main__":
    for key in ("c2", "c3", "c4"):
        wl = CONFIGS[key]
        for layer in range(wl.layers):
            a, s = calibrate(wl, layer)
            print(f'    ("{key}", {layer}): {a},   # top-20% share {s:.4f}')
