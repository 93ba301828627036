"""Test-side glue: drives one workload through the library's host planner and,
independently, through the oracle's planner.  Nothing here computes the
method; it only calls one side or the other."""

import math

import numpy as np

import oracle
import workloads as W
from position_independent_kv_stitch_gb300 import pic


def lib():
    return pic.load(build_if_missing=True) and pic


def spec_of(wl: W.Workload) -> pic.ModelSpec:
    return pic.model_spec_from(wl.model)


def oracle_theta(model: W.Model):
    return oracle.model_inv_freq(model.rope_dim, model.rope_theta, model.llama3)


def oracle_pairing(model: W.Model):
    return oracle.NEOX_HALF if model.pairing == "neox" else oracle.INTERLEAVED


def blocks_for(wl: W.Workload) -> int:
    bs = wl.model.block_size
    return sum(math.ceil(t / bs) for t in wl.request_tokens)


def max_blocks_for(wl: W.Workload) -> int:
    bs = wl.model.block_size
    return max(math.ceil(t / bs) for t in wl.request_tokens)


def lib_register(ctx, wl: W.Workload):
    ids = []
    for c, (off, n) in enumerate(zip(wl.pool_offsets, wl.chunk_lens)):
        cid, new = pic.pic_register_chunk(ctx, W.chunk_key(wl.name, c), off, n, 0)
        assert new
        ids.append(cid)
    return ids


def lib_plan(ctx, wl: W.Workload, ids, max_blocks=None):
    """Plans every request in order; returns (plans, block tables [n_req][max_blocks])."""
    max_blocks = max_blocks or max_blocks_for(wl)
    plans, tables = [], []
    for req in wl.requests:
        plan, bt = pic.pic_build_block_table(
            ctx, [ids[c] for c, _ in req], max_blocks, take_tokens=[t for _, t in req],
            k_nonleading=wl.k_nonleading, k_leading=wl.k_leading)
        plans.append(plan)
        tables.append(bt)
    return plans, np.stack(tables) if tables else np.zeros((0, max_blocks), np.int32)


def oracle_plan(wl: W.Workload, num_blocks: int):
    """Oracle plans: (segments per request, block tables as lists, recompute lists)."""
    chunks = [oracle.Chunk(off, n, 0) for off, n in zip(wl.pool_offsets, wl.chunk_lens)]
    pool = oracle.BlockPool(num_blocks)
    segs_all, tables, rec = [], [], []
    for req in wl.requests:
        segs = oracle.compose(chunks, [c for c, _ in req], take=[t for _, t in req])
        total = segs[-1].dst_pos + segs[-1].length if segs else 0
        tables.append(pool.allocate(oracle.blocks_needed(total, wl.model.block_size)))
        segs_all.append(segs)
        rec.append(oracle.recompute_positions(segs, wl.k_nonleading, wl.k_leading))
    return segs_all, tables, rec


def create_ctx(wl: W.Workload, num_blocks: int):
    return pic.create_from_spec(spec_of(wl), num_blocks)
