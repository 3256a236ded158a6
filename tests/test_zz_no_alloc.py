"""strata_route_topk_noalloc: the router entry point for callers that cannot allocate device memory
when they call in (e.g. enqueue steps of plugin interfaces, code running during CUDA graph
capture, processes whose memory belongs to one allocator). Its scratch is the library's own fixed
device array, so it must give exactly what strata_route_topk gives with a caller workspace —
checked here on two calls in a row with different shapes, through the C ABI.

This file is named to be collected last: a failure here leaves every other test already run.
"""
import numpy as np
import pytest

from workloads import CONFIGS, gen

pytestmark = pytest.mark.gpu


def _outputs(T, E, k):
    import torch
    z = lambda *shape, dt=torch.int32: torch.full(shape, -7, dtype=dt, device="cuda")  # noqa: E731
    return dict(ids=z(T, k), gates=z(T, k, dt=torch.float32), counts=z(E), offsets=z(E + 1),
                perm=z(T * k), inv=z(T, k))


def _route_both(key, T, seed_name):
    import torch
    import int4_grouped_expert_gb300 as st
    wl = CONFIGS[key]
    x = torch.from_numpy(gen.activations(T, wl.H, 0, name=seed_name).view(np.int16)).view(
        torch.bfloat16).cuda()
    wr = torch.from_numpy(gen.router_weight(wl)).cuda()
    b = gen.router_bias(wl)
    bias = None if b is None else torch.from_numpy(b).cuda()
    ref = _outputs(T, wl.E, wl.k)
    ws_bytes = st.strata_route_workspace_size(T, wl.E, wl.k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    st.check(st.strata_route_topk(x, wr, bias, T, wl.H, wl.E, wl.k, 0, workspace=ws,
                                  ws_bytes=ws_bytes, **ref), "strata_route_topk")
    got = _outputs(T, wl.E, wl.k)
    st.check(st.strata_route_topk_noalloc(x, wr, bias, T, wl.H, wl.E, wl.k, 0, **got),
             "strata_route_topk_noalloc")
    torch.cuda.synchronize()
    return {n: t.cpu().numpy() for n, t in ref.items()}, {n: t.cpu().numpy() for n, t in got.items()}


def _same(ref, got):
    for name in ("ids", "counts", "offsets", "perm", "inv"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)
    np.testing.assert_allclose(got["gates"], ref["gates"], rtol=1e-5, atol=0)


def test_noalloc_matches_workspace_router_on_two_calls():
    # first call: the 4096-token prefill router (the largest scratch these workloads need)
    ref, got = _route_both("c5", 4096, "noalloc/c5")
    _same(ref, got)
    # second call, different shape: the decode router with its Zipf bias; the array still holds
    # the first call's partial logits, which must not leak into this result
    ref, got = _route_both("c2", 16, "noalloc/c2")
    _same(ref, got)


def test_noalloc_rejects_requests_above_its_scratch():
    import int4_grouped_expert_gb300 as st
    T, E, k = 100_000, 64, 2          # router scratch alone: 100000 * 64 * 4 bytes > 8 MiB
    assert st.strata_route_workspace_size(T, E, k) > st.NOALLOC_SCRATCH_BYTES
    A = 1 << 12                       # never dereferenced: the size check comes first
    rc = st.strata_route_topk_noalloc(A, A, None, T, 1024, E, k, 0, A, A, A, A, A, A)
    assert rc == st.STATUS_NAMES.index("STRATA_ERR_UNSUPPORTED")
