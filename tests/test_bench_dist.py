"""bench.py's multi-rank plumbing on CPU: two gloo ranks agree on the max step time and
the summed row count (weak scaling, replicas; no data-path collective exists)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    t = bench.reduce_max(10.0 + 5.0 * rank, w)
    rows = bench.reduce_sum(64.0 * (rank + 1), w)
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((r, w, t, rows))


def test_two_rank_timing_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1]
    for _, w, t, rows in res:
        assert w == 2 and t == 15.0 and rows == 192.0


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.reduce_sum(7.0, 1) == 7.0


def test_launch_distribution_summary():
    sys.path.insert(0, ROOT)
    import bench
    d = bench.launch_dist([0.05, 0.01, 0.02, 0.03, 0.04, 0.06, 0.07, 0.08, 0.09, 0.10, 0.11])
    assert d == {"median": 60.0, "p10": 20.0, "p90": 100.0}
    assert bench.launch_dist([0.042]) == {"median": 42.0, "p10": 42.0, "p90": 42.0}
    assert bench.launch_dist([]) is None
