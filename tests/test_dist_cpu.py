"""The benchmark's multi-process glue on CPU: two gloo ranks (127.0.0.1) run the same
barrier and max-over-ranks timing reduction that bench.py uses for --gpus N (one
independent replica of the workload per GPU, no collective on the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    # each replica reports its own elapsed time; the job's time is the slowest rank's
    t = d.max(10.0 + 5.0 * rank)
    d.barrier()
    out_q.put((rank, d.world, t))
    d.close()


@pytest.mark.parametrize("world", [2])
def test_dist_barrier_and_max_over_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[0] for r in res] == list(range(world))
    assert all(r[1] == world for r in res)
    assert all(r[2] == 10.0 + 5.0 * (world - 1) for r in res)
