"""The multi-rank host path of bench.py on CPU: two gloo ranks.

Under torchrun every rank runs its own replica of the round (no data-path
collective); the only cross-rank steps are the barrier around the timed
region and the max over ranks of the per-rank time. Both are exercised here
with world size 2 on the gloo backend, through bench.py's own helpers.
"""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench

    class Args:
        pass

    w, r, local = bench.dist_init(Args())
    bench.barrier(w)
    t = bench.max_over_ranks(1.0 + 2.0 * rank, w)   # per-rank "times" 1.0 and 3.0
    bench.barrier(w)
    results[rank] = (w, r, local, t)
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.skipif(not torch.distributed.is_available(), reason="torch.distributed missing")
@pytest.mark.skipif(torch.cuda.is_available(), reason="the gloo path is the CPU one; a GPU box runs nccl ranks")
def test_two_gloo_ranks_agree_on_the_max_time():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
        assert p.exitcode == 0
    assert sorted(results.keys()) == [0, 1]
    for rank in range(world):
        w, r, local, t = results[rank]
        assert (w, r, local) == (world, rank, rank)
        assert t == 3.0                                # every rank sees the slowest rank's time
