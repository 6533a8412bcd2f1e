"""The bench's multi-rank path on CPU: two gloo ranks run the timed loop
(barrier + sync on both sides of exactly K steps) and agree on the maximum
over ranks, which is what the JSON line reports for N > 1 replicas."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import time
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist = bench.Dist(backend="gloo")
    steps, warmup = 4, 3
    calls = {"step": 0, "flush": 0}
    delay = 0.01 * (rank + 1)

    def step():
        calls["step"] += 1
        time.sleep(delay)

    def flush():
        calls["flush"] += 1

    total_max, per = bench.timed_loop(dist, steps, warmup, step, flush, bench.WallTimer(), lambda: None)
    total_sum = dist.sum(sum(per))
    q.put((rank, total_max, sum(per), len(per), calls["step"], calls["flush"], total_sum))
    dist.close()


def test_two_rank_timed_loop_max_over_ranks():
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
    (r0, max0, loc0, n0, s0, f0, sum0), (r1, max1, loc1, n1, s1, f1, sum1) = res
    assert n0 == n1 == 4                      # exactly K timed steps
    assert s0 == s1 == 7 and f0 == f1 == 7   # K + W steps, one flush before each
    assert max0 == max1 == pytest.approx(max(loc0, loc1))
    assert loc1 > loc0                        # rank 1 sleeps twice as long
    assert sum0 == sum1 == pytest.approx(loc0 + loc1)
