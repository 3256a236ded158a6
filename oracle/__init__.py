"""Oracle for the routed int4-g128 MoE layer: plain, slow, fp64 NumPy.

TEST INFRASTRUCTURE ONLY. Only `tests/`, `__graft_entry__.smoke()` and the CPU
baseline legs of `bench.py` may import this package. The library
(`int4_grouped_expert_gb300`) never imports it, and this package imports
nothing from the library: the two share no kernels, headers, helpers or
constants. Inputs come from `workloads` (seeded generators, no method
arithmetic).

Every function states the write-up passage it follows. The pages print no
worked numeric example, so each function is pinned instead by closed forms,
invariants, special cases and brute force (tests/test_oracle_*.py).

Functions and their pins:
  quantize_groups   pinned: exact-rational brute force, |w - q s| <= s/2,
                    absmax -> +-7 (+-127 for 8 bits), idempotence, hand-built
                    .5 ties (golden), for 4- and 8-bit codes.
  dequantize        pinned: hand-packed bytes (golden) and round trip.
  route_topk        pinned: pure-Python brute force, full sort, sum p = 1,
                    k = E, zero router -> uniform.
  permute           pinned: brute-force stable sort, bijection, counts.
  expert_ffn /
  moe_forward       pinned: pure-Python loops on tiny shapes, dense
                    equivalence (k = E, zero router), E = k = 1, token
                    independence.
Nothing in this package is "parity unpinned".
"""
from .strata_oracle import (  # noqa: F401
    GROUP,
    bf16_to_f64,
    dequantize,
    expert_ffn,
    moe_forward,
    pack_codes,
    permute,
    quantize_groups,
    quantize_groups_f16_quotient,
    route_topk,
    unpack_codes,
)
