"""The request-split batch's host logic on CPU: ranges and the one exchange.

A batch split by request across devices plans the whole batch on every
device, because the planner prices the whole verify batch (SPS of the total
verify tokens). The exchange that makes this possible is an all-gather of
every rank's confidences; two gloo ranks run it here through
``shard.gather_confidences`` on uneven shares, then each plans the gathered
batch and keeps its own range. The concatenated per-rank lengths must equal
the plan of the unsplit batch. The planner here is the fp64 oracle (the
library's planner and its slicing kernel need a GPU and are held to the
unsplit batch in the GPU tests); what is under test is the split, the gather
and the bookkeeping around them.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from speculative_decoding_head_gb300 import shard
from speculative_decoding_head_gb300.workloads import WORKLOADS, sps_table

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_shard_ranges_cover_the_batch_in_order():
    for B in (1, 2, 7, 41, 128, 257):
        for world in range(1, min(B, 9) + 1):
            counts = shard.shard_counts(B, world)
            assert sum(counts) == B and max(counts) - min(counts) <= 1
            assert counts == sorted(counts, reverse=True)
            nxt = 0
            for rank in range(world):
                b0, n = shard.shard_range(B, rank, world)
                assert b0 == nxt and n == counts[rank] and n >= 1
                nxt = b0 + n
            assert nxt == B
    with pytest.raises(ValueError):
        shard.shard_counts(3, 4)          # a rank with no request
    with pytest.raises(ValueError):
        shard.shard_range(8, 2, 2)


def test_single_rank_gather_is_the_identity():
    conf = torch.rand(5, 3)
    assert shard.gather_confidences(conf, 5, 0, 1) is conf
    with pytest.raises(ValueError):
        shard.gather_confidences(conf, 6, 0, 1)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


# 41 requests over two ranks: shares of 21 and 20, so the gather pads one rank
WL = WORKLOADS["prod"].with_(B=41, sps_knee=24.0)


def _confidences(rnd):
    g = torch.Generator().manual_seed(1000 + rnd)
    # a spread of per-request confidence levels, falling along the block
    base = torch.rand(WL.B, 1, generator=g) * 0.6 + 0.35
    return (base * (1.0 - 0.05 * torch.rand(WL.B, WL.gamma, generator=g))).to(torch.float32)


def _rank_main(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist

    import oracle
    from speculative_decoding_head_gb300 import shard as sh

    dist.init_process_group("gloo", rank=rank, world_size=world)
    b0, n = sh.shard_range(WL.B, rank, world)
    sps = sps_table(WL).numpy()
    out = []
    for rnd in range(3):
        conf_all = _confidences(rnd)
        mine = conf_all[b0:b0 + n].clone()
        got = sh.gather_confidences(mine, WL.B, rank, world)
        L, _, _ = oracle.plan_sync(got.numpy(), sps)
        out.append((bool(torch.equal(got, conf_all)), L[b0:b0 + n].tolist()))
    results[rank] = out
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.skipif(not torch.distributed.is_available(), reason="torch.distributed missing")
def test_two_gloo_ranks_plan_the_gathered_batch_like_one_process():
    import oracle

    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    sps = sps_table(WL).numpy()
    for rnd in range(3):
        whole, _, pm = oracle.plan_sync(_confidences(rnd).numpy(), sps)
        assert not pm.flagged(1e-9, 1e-9)
        parts = []
        for rank in range(world):
            gathered_ok, lengths = results[rank][rnd]
            assert gathered_ok, (rank, rnd)
            parts += lengths
        assert parts == whole.tolist(), rnd
        # the planner must actually shorten some requests for the check to bite
        assert (whole < WL.gamma + 1).any() and (whole > 1).any()
