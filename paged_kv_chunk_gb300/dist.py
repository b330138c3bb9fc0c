"""Multi-rank plumbing for running the path on several GPUs of one node.

The path shards with no exchange (ASR Engine page, section 4.3: streams are independent, each
owns its block table, pool slice and output rows; heads and packed utterances likewise), so
ranks share nothing on the data path.  What crosses ranks is host-side only: the rank layout,
a barrier around timed regions, the slowest rank's time, and how work is split.

* ``setup()`` reads RANK / WORLD_SIZE / LOCAL_RANK and joins the process group (NCCL when the
  rank has a GPU, gloo otherwise; rendezvous from MASTER_ADDR / MASTER_PORT).
* ``stream_shard(B, world, rank)``: the rank's contiguous range of a cohort's streams.
* ``balance_segments(lengths, world)``: packed utterances split into per-rank bins of near
  equal attention cost (sum of L^2), longest first onto the lightest bin.
* ``barrier()`` and ``max_over_ranks(x)`` for timing.
"""
from __future__ import annotations

import os

import numpy as np
import torch


def env_ranks():
    """(rank, world, local_rank) from the launcher's environment (1 rank when unset)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _dist():
    import torch.distributed as dist
    return dist


def setup(backend: str | None = None):
    """Join the process group when WORLD_SIZE > 1 and pick this rank's GPU; returns
    (rank, world, local_rank)."""
    rank, world, local = env_ranks()
    use_cuda = torch.cuda.is_available()
    if use_cuda:
        torch.cuda.set_device(local if world > 1 else 0)
    if world > 1:
        dist = _dist()
        if not dist.is_initialized():
            dist.init_process_group(backend or ("nccl" if use_cuda else "gloo"))
    return rank, world, local


def _world():
    dist = _dist()
    return dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1


def barrier():
    if _world() > 1:
        _dist().barrier()


def max_over_ranks(x: float) -> float:
    """The largest x over all ranks (the slowest rank's time)."""
    if _world() == 1:
        return float(x)
    dist = _dist()
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def stream_shard(B: int, world: int, rank: int) -> range:
    """Contiguous streams [lo, hi) of rank `rank` when B streams are split over `world` ranks
    (sizes differ by at most one)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    base, extra = divmod(B, world)
    lo = rank * base + min(rank, extra)
    return range(lo, lo + base + (1 if rank < extra else 0))


def balance_segments(lengths, world: int) -> list[list[int]]:
    """Per-rank lists of segment indices (each in ascending order) whose attention costs
    (sum of L^2) are near equal: segments are taken longest first and each goes to the bin
    with the least cost so far (ties to the lower rank).  The heaviest bin exceeds the mean by
    at most the largest single segment's cost."""
    if world < 1:
        raise ValueError("world must be >= 1")
    lengths = np.asarray(lengths, dtype=np.int64)
    cost = lengths * lengths
    bins = [[] for _ in range(world)]
    load = np.zeros(world, dtype=np.int64)
    for s in sorted(range(len(lengths)), key=lambda i: (-cost[i], i)):
        r = int(np.argmin(load))
        bins[r].append(s)
        load[r] += cost[s]
    return [sorted(b) for b in bins]


def pack_subset(x: dict, segs: list[int]) -> dict:
    """The packed inputs of the segments `segs` (rows gathered, cu_seqlens rebuilt); the rel
    table and biases are shared."""
    cu = np.asarray(x["cu_seqlens"])
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in segs]) if segs else np.zeros(0, np.int64)
    lens = np.array([cu[s + 1] - cu[s] for s in segs], dtype=np.int32)
    out = dict(x)
    for k in ("q", "k", "v"):
        out[k] = x[k][rows]
    out["cu_seqlens"] = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out["lengths"] = lens
    out["max_seqlen"] = int(lens.max()) if len(lens) else 0
    return out
