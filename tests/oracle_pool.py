"""The oracle's layer output for many tokens at once (test infrastructure).

A token's output needs every expert it is routed to, and a few hundred tokens of a large layer
reach nearly all experts; the oracle's expert work (regenerate the fp16 weights, quantize,
dequantize, run the FFN on the expert's rows) is then spread over worker processes, one expert
per job. The workers run only the oracle's own functions, and the routing and the weighted
combine stay in oracle.moe_forward (expert_out). Workers are started with "spawn": a pool
forked after the first GPU call would hang.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _expert_rows(job):
    wl, layer, e, x_bits, group, bits = job
    import oracle
    from workloads import gen
    mats = gen.expert_weights(wl, e, layer)
    w = [oracle.dequantize(*oracle.quantize_groups(m, group=group, bits=bits)) for m in mats]
    return e, oracle.expert_ffn(oracle.bf16_to_f64(x_bits), *w)


def moe_forward(wl, x_bits, w_router, bias, tokens, layer=0, residual=False, renorm=False,
                group=128, bits=4, procs=None):
    """oracle.moe_forward on the given tokens, the experts evaluated in worker processes."""
    import oracle
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    tokens = np.asarray(tokens)
    xs = x_bits[tokens]
    ids = oracle.route_topk(xs, w_router, bias, wl.k, renorm=renorm)["ids"]
    jobs = []
    for e in np.unique(ids):
        rows = np.argwhere(ids == e)[:, 0]     # the order oracle.moe_forward uses
        jobs.append((wl, layer, int(e), xs[rows], group, bits))
    if wl.shared:
        jobs.append((wl, layer, wl.E, xs, group, bits))
    jobs.sort(key=lambda j: -len(j[3]))
    n = max(1, min(len(jobs), procs or os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(n) as pool:
        out = dict(pool.imap_unordered(_expert_rows, jobs, chunksize=1))
    return oracle.moe_forward(x_bits, w_router, bias, wl.k, None, wl.E, wl.shared, renorm=renorm,
                              residual=residual, tokens=tokens, expert_out=out)
