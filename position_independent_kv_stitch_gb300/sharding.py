"""Sharding of stitch work across ranks (one process per GPU).

Stitching has no exchange step: every request (and every layer and KV head
of it) is independent.  Ranks therefore split a batch by request (data
parallel) or hold a share of every request's KV heads (tensor parallel, as
the EPIC guide's deployment runs it with 4 GPUs) and never talk on the data
path; the only collective is the benchmark's max-over-ranks timing.
"""

from __future__ import annotations


def shard_requests(n_requests: int, rank: int, world: int):
    """Contiguous, balanced request range [lo, hi) owned by `rank`."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    base, extra = divmod(n_requests, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def shard_kv_heads(n_kv_heads: int, rank: int, world: int):
    """KV heads [lo, hi) held by `rank` under tensor parallelism.

    Each rank holds whole heads, n_kv_heads / world of them, in its own pool
    and cache ([L][tokens][heads of this rank][head_dim]).  The RoPE shift
    acts on each head by itself, so every rank stitches its heads with the
    same host plan (the same block table and recompute list) and no rank
    needs another's data.
    """
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    if n_kv_heads <= 0 or n_kv_heads % world:
        raise ValueError("KV heads must split evenly across the ranks")
    per = n_kv_heads // world
    return rank * per, (rank + 1) * per


def max_over_ranks(value: float, device=None) -> float:
    """Max of a float over all ranks of the default process group (identity
    without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
