"""The bench's N > 1 host logic on CPU: two gloo ranks, each with its own batch (weak
scaling, no data exchange), a barrier, the max-over-ranks step time and the whole-job
rate from it."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup(None, backend="gloo")
    try:
        bench.barrier(w)
        # Rank r's step took (r + 1) ms: the job's step time is the slowest rank's.
        slow = bench.max_over_ranks(float(r + 1), w)
        rate = bench.whole_job_rate(1_000_000_000, w, slow)
        q.put((r, w, local, slow, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [x[0] for x in res] == [0, 1]
    for r, w, local, slow, rate in res:
        assert w == 2 and local == r
        assert slow == 2.0                    # max over ranks, seen by every rank
        assert rate == pytest.approx(1000.0)  # 2 ranks x 1 GB in 2 ms = 1000 GB/s


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(2_000_000_000, 1, 4.0) == pytest.approx(500.0)
