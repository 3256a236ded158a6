"""Error paths on the GPU, in forms that fault, trap or hang nothing.

- Bounded waits: strata_selftest_bounded_waits runs the library's mbarrier wait (the TMA-fed
  grouped GEMMs) and counter spin (the fused router) on a barrier and a counter that nothing
  completes, with a short limit. Both must give up, flag STRATA_DEV_TIMEOUT and return; the status
  read then returns STRATA_ERR_TIMEOUT, and the context serves a correct layer afterwards.
- Bad expert ids: strata_group_rows (the grouping step of "Strata" 3090 tuning,
  xdnf.cn/news/329730, §3.2) on caller-given ids is exact against the oracle's permutation, and
  ids outside [0, E) set STRATA_DEV_BAD_ID, are left out of every group (inv = -1) and leave the
  valid rows where the oracle puts them.
"""
import time

import numpy as np
import pytest

import oracle
from helpers import OracleExperts, build_gpu_layer, compare_output, compare_routing, run_forward
from workloads import CONFIGS, gen

pytestmark = pytest.mark.gpu


def test_bounded_waits_give_up_and_report_a_timeout():
    import torch
    import int4_grouped_expert_gb300 as st
    words = torch.zeros(4, dtype=torch.int32, device="cuda")
    limit = 20_000_000                      # SM clocks: ~10 ms at 2 GHz, per wait
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st.check(st.strata_selftest_bounded_waits(words, limit), "selftest")
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    w = words.cpu().numpy().view(np.uint32)
    assert w[1] == 0, "nothing may increment the counter"
    assert w[2] == 1, "the mbarrier wait did not give up"
    assert w[3] == 1, "the counter spin did not give up"
    assert dt < 5.0, f"the waits took {dt:.2f} s"
    rc, v = st.strata_read_status(words)
    assert rc == st.STRATA_ERR_TIMEOUT, st.strata_status_string(rc)
    assert v == st.STRATA_DEV_TIMEOUT
    # the status word was cleared by the read, and the context is still good for real work
    assert st.strata_read_status(words) == (0, 0)
    wl = CONFIGS["c1"]
    L, wr, b = build_gpu_layer(wl)
    x = gen.activations(8, wl.H, wl.seed, name="after_timeout")
    got = run_forward(L, x)
    ref = oracle.moe_forward(x, wr, b, wl.k, OracleExperts(wl), wl.E, wl.shared)
    diff, _ = compare_routing(got, ref["route"], wl.E)
    compare_output(got["out"][~diff], ref["out"][~diff])


def group_on_gpu(ids, E):
    import torch
    import int4_grouped_expert_gb300 as st
    T, k = ids.shape
    d = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(st.GROUP_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    st.check(st.strata_group_rows(d, T, k, E, counts, offsets, perm, inv, ws, ws.numel()), "group")
    rc, v = st.strata_workspace_status(ws)
    return (dict(counts=counts.cpu().numpy(), offsets=offsets.cpu().numpy(),
                 perm=perm.cpu().numpy(), inv=inv.cpu().numpy()), rc, v)


@pytest.mark.parametrize("T,k,E", [(300, 8, 288), (4096, 8, 256), (1, 1, 1), (37, 32, 1024),
                                   (64, 4, 5)])
def test_group_rows_matches_the_oracle(T, k, E):
    rng = np.random.default_rng(T * 1000 + k)
    # distinct experts per token (as a router gives) for the first half, repeats allowed after
    ids = np.stack([rng.choice(E, k, replace=False) if (t < T // 2 and k <= E)
                    else rng.integers(0, E, k) for t in range(T)]).astype(np.int32)
    got, rc, v = group_on_gpu(ids, E)
    assert rc == 0, f"device status 0x{v:x}"
    ref = oracle.permute(ids, E)
    for name in ("counts", "offsets", "perm", "inv"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)


def test_group_rows_empty_batch():
    got, rc, _ = group_on_gpu(np.zeros((0, 4), dtype=np.int32), 16)
    assert rc == 0
    assert (got["counts"] == 0).all() and (got["offsets"] == 0).all()


def test_bad_ids_are_flagged_and_left_out():
    import int4_grouped_expert_gb300 as st
    T, k, E = 300, 8, 288
    rng = np.random.default_rng(7)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    bad = [(3, 2, -1), (100, 0, E), (299, 7, 1 << 30), (150, 4, -(1 << 31))]
    for t, j, val in bad:
        ids[t, j] = val
    got, rc, v = group_on_gpu(ids, E)
    assert rc == st.STRATA_ERR_DEVICE_STATUS and v == st.STRATA_DEV_BAD_ID, (rc, hex(v))
    # expected: the oracle's grouping with every bad row sent to one extra expert E, which sorts
    # after all valid ones, so the valid rows keep the positions they have without the bad ones
    ids_x = ids.copy()
    mask = np.zeros((T, k), dtype=bool)
    for t, j, _ in bad:
        ids_x[t, j] = E
        mask[t, j] = True
    ref = oracle.permute(ids_x, E + 1)
    n_valid = T * k - len(bad)
    np.testing.assert_array_equal(got["counts"], ref["counts"][:E])
    np.testing.assert_array_equal(got["offsets"], ref["offsets"][:E + 1])
    assert got["offsets"][E] == n_valid
    np.testing.assert_array_equal(got["perm"][:n_valid], ref["perm"][:n_valid])
    np.testing.assert_array_equal(got["inv"][~mask], ref["inv"][~mask])
    assert (got["inv"][mask] == -1).all()
