"""The multi-rank side of bench.py on CPU: two gloo ranks (one process each, as torchrun starts them)
check the rendezvous, the barrier, the max-over-ranks time and the whole-job throughput that the
benchmark reports for N replicas of the layer."""
import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    try:
        import torch.distributed as dist
        import bench
        ws, r = bench.init_dist("gloo")
        bench.barrier()
        slowest = bench.max_over_ranks(1.0 + rank)          # rank 1 is the slow one: 2.0 s
        value = bench.aggregate_throughput(100, 1.0 + rank, ws)
        bench.barrier()
        dist.destroy_process_group()
        q.put((rank, ws, r, slowest, value, None))
    except Exception as exc:  # noqa: BLE001 - reported to the parent
        q.put((rank, None, None, None, None, repr(exc)))


def test_two_gloo_ranks_aggregate_like_the_benchmark():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    res.sort()
    for rank, ws, r, slowest, value, err in res:
        assert err is None, err
        assert (ws, r) == (2, rank)
        assert slowest == pytest.approx(2.0)       # the max over ranks, seen by every rank
        assert value == pytest.approx(100.0)       # 2 ranks x 100 tokens / 2.0 s


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.init_dist("gloo") == (1, 0)
        assert bench.max_over_ranks(3.5) == 3.5
        assert bench.aggregate_throughput(16, 0.5, 1) == pytest.approx(32.0)
    finally:
        os.environ.update(env)
