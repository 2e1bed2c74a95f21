"""The multi-process path of bench.py on the CPU: two ranks over gloo.

Every rank verifies its own batch (independent replicas, no collective on
the data path); the only cross-rank steps are the barrier around the timed
region and the reductions of the timings (max over ranks) and of the work
done (sum over ranks), which this test checks."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks()
    try:
        r.barrier()
        t = r.max(10.0 + rank)          # slowest rank's time
        w = r.sum(100.0 * (rank + 1))   # work of all ranks
        out.put((rank, t, w))
    finally:
        r.close()


@pytest.mark.timeout(120)
def test_two_ranks_reduce_time_and_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert res == [(0, 11.0, 300.0), (1, 11.0, 300.0)]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    saved = {k: os.environ.pop(k, None) for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    try:
        r = bench.Ranks()
        assert r.world == 1 and r.dist is None
        assert r.max(3.5) == 3.5 and r.sum(2.0) == 2.0
        r.barrier()
    finally:
        for k, v in saved.items():
            if v is not None:
                os.environ[k] = v
