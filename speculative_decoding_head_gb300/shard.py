"""A DSpark batch split by request across devices, one process per GPU.

Draft and verify treat every request on its own. The planner does not: its
objective Theta = tau * SPS(B_tot) ("spec_dspark", section "目标函数") prices
the target engine's whole verify batch, so one request's length depends on
every request's confidences. A round over a split batch therefore has one
exchange step: before planning, every device all-gathers the B_local x gamma
fp32 confidences of the others (B * gamma * 4 bytes in all). Each device
then runs the same deterministic planner on the same gathered confidences,
keeps its own range of lengths, and verifies its own requests. Random draws
key on a request's index in the whole batch, so a request draws the same
numbers wherever it runs, and the split round returns exactly what one
device would return for the whole batch.

Everything here is marshalling; the planner, the slicing of its output and
every draw run in libdspark's kernels.
"""

from __future__ import annotations

from typing import List, Optional, Tuple

import torch

from .binding import Workspace


def shard_counts(B: int, world: int) -> List[int]:
    """Requests per rank: contiguous ranges, the first B % world ranks one longer."""
    if world < 1 or B < world:
        raise ValueError(f"cannot split {B} requests over {world} ranks")
    q, m = divmod(B, world)
    return [q + (1 if i < m else 0) for i in range(world)]


def shard_range(B: int, rank: int, world: int) -> Tuple[int, int]:
    """(b_begin, b_count) of ``rank``'s requests in a batch of B."""
    counts = shard_counts(B, world)
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world {world}")
    return sum(counts[:rank]), counts[rank]


def gather_confidences(conf_local: torch.Tensor, B: int, rank: int, world: int, group=None) -> torch.Tensor:
    """All-gather every rank's confidences [b_count, gamma] into [B, gamma] in
    batch order. Ranks hold unequal counts, so each sends its rows padded to
    the largest count and the pads are dropped after the gather. A single
    process (world 1) returns its own rows."""
    counts = shard_counts(B, world)
    if conf_local.dim() != 2 or conf_local.shape[0] != counts[rank]:
        raise ValueError(f"rank {rank} holds {counts[rank]} requests, got confidences {tuple(conf_local.shape)}")
    if world == 1:
        return conf_local
    import torch.distributed as dist

    n = max(counts)
    g = conf_local.shape[1]
    send = torch.zeros((n, g), dtype=conf_local.dtype, device=conf_local.device)
    send[:counts[rank]] = conf_local
    recv = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(recv, send, group=group)
    return torch.cat([t[:c] for t, c in zip(recv, counts)], dim=0).contiguous()


class ShardedRound:
    """One rank's part of a request-split round: a workspace for its own
    requests (draft and verify, the draws keyed by batch index) and one for
    the whole batch (the planner, whose ring of lagged capacities every rank
    keeps in step because every rank plans the same confidences)."""

    def __init__(self, B: int, gamma: int, V: int, r: int, H: int, wdtype: str = "bf16",
                 mode: str = "compact", lag: int = 2, rank: int = 0, world: int = 1, group=None,
                 path: Optional[str] = None):
        self.B, self.rank, self.world, self.group = B, rank, world, group
        self.b_begin, self.b_count = shard_range(B, rank, world)
        self.local = Workspace(self.b_count, gamma, V, r, H, wdtype, mode, lag, path)
        self.local.set_shard(self.b_begin)
        self.planner = Workspace(B, gamma, V, r, H, wdtype, mode, lag, path)

    def draft(self, U, W1, W2, anchor, h, w, T, seed: int, rnd: int, out=None, stream=None):
        """Draft this rank's requests (inputs hold only them)."""
        return self.local.draft(U, W1, W2, anchor, h, w, T, seed, rnd, out=out, stream=stream)

    def plan(self, conf_local, sps, out=None, stream=None):
        """Gather the batch's confidences, plan the whole batch, keep this
        rank's lengths ("lengths_local") and packed-row offsets ("row_off_local")."""
        conf = gather_confidences(conf_local, self.B, self.rank, self.world, self.group)
        return self.planner.plan_shard(conf, sps, self.b_begin, self.b_count, out=out, stream=stream)

    def verify(self, P, row_off_local, lengths_local, anchor, tokens, pd_tok, lse, U, W1, W2, seed: int, rnd: int,
               out=None, stream=None):
        """Verify this rank's requests on its own packed target rows."""
        return self.local.verify(P, row_off_local, lengths_local, anchor, tokens, pd_tok, lse, U, W1, W2, seed,
                                 rnd, out=out, stream=stream)

    def close(self) -> None:
        self.local.close()
        self.planner.close()
