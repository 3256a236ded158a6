"""The five synthetic workloads of the routed int4-g128 MoE layer.

Shapes follow the engine write-ups' problem statement: a router picks k of E
experts per token ("Strata" tuning notes, lpnh.cn/news/2730718, §3.3 config
dict, routing_top_k), expert FFNs are Gate/Up + Down ("GLM-5.3-Flash on one
4090", haowenji.com, §01) and a shared expert is always on (same page, §01:
8 routed experts plus 1 shared per token). The pages measure on private models
and traces; these seeded shapes and distributions stand in for them.

Notation: T tokens, H hidden, I expert intermediate size, E routed experts,
k experts per token, S = 1 when a shared expert (index E) is present.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Tuple


@dataclass(frozen=True)
class Workload:
    key: str
    name: str
    H: int
    I: int
    E: int
    k: int
    shared: int
    batches: Tuple[int, ...]
    router: str                 # "uniform" (N(0,0.02), no bias) or "zipf"
    layers: int = 1
    router_variants: Tuple[str, ...] = field(default_factory=tuple)
    seed: int = 0
    quantize_on_device: bool = True

    @property
    def n_experts_total(self) -> int:
        return self.E + self.shared

    def expert_bytes(self) -> int:
        """int4 codes + fp16 scales of one expert's three matrices."""
        n = 3 * self.H * self.I
        return n // 2 + 2 * (n // 128)


CONFIGS = {
    "c1": Workload("c1", "single_moe_layer_h1024_e16_top2", H=1024, I=512, E=16, k=2,
                   shared=0, batches=(64,), router="uniform"),
    "c2": Workload("c2", "decode_moe_layer_h4096_e288_top8_shared", H=4096, I=1536, E=288,
                   k=8, shared=1, batches=(1, 4, 8, 16), router="zipf"),
    "c3": Workload("c3", "prefill_moe_layer_h5120_e64_top4", H=5120, I=2048, E=64, k=4,
                   shared=0, batches=(512,), router="uniform", router_variants=("zipf",)),
    "c4": Workload("c4", "decode_moe_stack8_h4096_e128_top4_shared", H=4096, I=2048, E=128,
                   k=4, shared=1, batches=(1, 4, 8, 16, 32), router="zipf", layers=8),
    "c5": Workload("c5", "prefill_quantize_layer_h7168_e256_top8_shared", H=7168, I=2048,
                   E=256, k=8, shared=1, batches=(4096,), router="uniform"),
}

# Zipf(s=1.1) router bias strength alpha, per (config, layer): bias_e = alpha * ln p_rank(e).
# Each alpha was found by seeded bisection (tests/golden/calibrate_zipf.py, which
# routes a separate 2048-token calibration batch with the oracle) so that the
# 20% most-used experts take 80% +- 1% of the routes; tests/test_workloads.py
# re-checks the share for every entry. The pages' own statistic: the top 20% of
# experts take 80%+ of activations ("Strata" 3090 tuning, xdnf.cn/news/329730, §2.1).
ZIPF_S = 1.1
ZIPF_ALPHA = {
    ("c2", 0): 0.68744,
    ("c3", 0): 1.064587,
    ("c4", 0): 0.744875, ("c4", 1): 0.736987, ("c4", 2): 0.731733, ("c4", 3): 0.740268,
    ("c4", 4): 0.736774, ("c4", 5): 0.751118, ("c4", 6): 0.726124, ("c4", 7): 0.749724,
}


def get(key: str) -> Workload:
    return CONFIGS[key]
