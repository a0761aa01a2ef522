"""Sharding a KV cache across ranks by layer, and stitching the bitstreams.

Chunks are independent (SKV v1 format §7), so the coder shards with no
data-path exchange: each rank codes a contiguous range of layers as a layout
of its own, and the one global bitstream is the ranks' streams back to back.
The only exchange is an exclusive scan of the per-rank byte totals, which
turns each rank's local offsets into global ones.

Host logic only; with torch.distributed it works on any backend (the tests
run it with gloo on CPU).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class LayerRange:
    rank: int
    first: int      # first layer of this rank
    count: int      # number of layers (may be 0)


def layer_ranges(n_layers: int, world: int) -> list[LayerRange]:
    """Contiguous, balanced layer ranges: the first n_layers % world ranks get one more."""
    if world < 1:
        raise ValueError("world must be >= 1")
    base, extra = divmod(n_layers, world)
    out, first = [], 0
    for r in range(world):
        cnt = base + (1 if r < extra else 0)
        out.append(LayerRange(r, first, cnt))
        first += cnt
    return out


def global_offsets(local_offsets: torch.Tensor, base: int) -> torch.Tensor:
    """Local offsets (n_local + 1, starting at 0) shifted to the rank's byte base."""
    return local_offsets.to(torch.int64) + int(base)


def exclusive_bases(totals: list[int]) -> list[int]:
    """Byte base of each rank: exclusive prefix sum of the per-rank totals."""
    out, acc = [], 0
    for t in totals:
        out.append(acc)
        acc += int(t)
    return out


def stitch(local_streams: list[torch.Tensor], local_offsets: list[torch.Tensor]):
    """One bitstream and offset table from per-rank (stream, offsets), in rank order."""
    totals = [int(o[-1]) for o in local_offsets]
    bases = exclusive_bases(totals)
    offs = [global_offsets(o[:-1], b) for o, b in zip(local_offsets, bases)]
    offs.append(torch.tensor([sum(totals)], dtype=torch.int64))
    return torch.cat([s.reshape(-1) for s in local_streams]), torch.cat(offs)


def distributed_base(local_total: int, group=None, device=None) -> tuple[int, int]:
    """(this rank's byte base, global total) via an all-gather of the totals
    (device: where the collective's tensors live, e.g. the rank's GPU for NCCL)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    t = torch.tensor([int(local_total)], dtype=torch.int64, device=device)
    got = [torch.zeros(1, dtype=torch.int64, device=device) for _ in range(world)]
    dist.all_gather(got, t, group=group)
    totals = [int(x.item()) for x in got]
    return exclusive_bases(totals)[dist.get_rank(group)], sum(totals)


def allreduce_counts(local_counts: torch.Tensor, group=None) -> torch.Tensor:
    """The global code histogram (p_hat's counts) from each rank's own layers."""
    import torch.distributed as dist
    c = local_counts.to(torch.int64).clone()
    dist.all_reduce(c, op=dist.ReduceOp.SUM, group=group)
    return c


def rank_inputs(cache: dict, rank: int, world: int, histogram, group=None):
    """This rank's share of one cache and the global code histogram.

    cache: {"kv", "mu", "sigma"} with the layer as the outermost dimension
    (the canonical [L][n_kv][T][H][D] codes and [L][n_kv][H][D] sigma).
    histogram(kv_part) -> int64 counts of the rank's own codes (on the device
    the collective runs on). Returns (LayerRange, {"kv", "mu", "sigma"} views
    of the rank's layers, global counts): the counts are all-reduced, since
    p_hat is one global table both ends hold.
    """
    n_layers = cache["kv"].shape[0]
    rng = layer_ranges(n_layers, world)[rank]
    sl = slice(rng.first, rng.first + rng.count)
    part = {k: cache[k][sl] for k in ("kv", "mu", "sigma")}
    local = histogram(part["kv"])
    counts = allreduce_counts(local, group) if world > 1 else local.to(torch.int64)
    return rng, part, counts
