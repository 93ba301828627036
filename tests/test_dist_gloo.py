"""World-size-2 CPU tests of the multi-GPU path, gloo backend, no GPU.
Data parallel: ranks split a batch by request, plan their share through the
C ABI's host side and agree with the oracle on it; the shards cover the
batch exactly once; timing is reduced with a max over ranks.  Tensor
parallel: ranks hold halves of the KV heads, plan the same request to the
same block table and recompute list, and each rank's stitched heads are its
share of the full stitch."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, errq):
    try:
        import sys
        sys.path.insert(0, ROOT)
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle
        import workloads as W
        from harness import lib
        from position_independent_kv_stitch_gb300 import pic
        from position_independent_kv_stitch_gb300.sharding import max_over_ranks, shard_requests
        lib()
        wl = W.qwen3_8b_batch(n_requests=5, request_tokens=4096)
        lo, hi = shard_requests(len(wl.requests), rank, world)
        mine = W.Workload(wl.name, wl.model, wl.chunk_lens, wl.requests[lo:hi], wl.k_nonleading, wl.k_leading)
        bs = wl.model.block_size
        nb = sum(-(-t // bs) for t in mine.request_tokens)
        ctx = pic.create_from_spec(pic.model_spec_from(wl.model), nb)
        ids = [pic.pic_register_chunk(ctx, W.chunk_key(wl.name, c), off, n)[0]
               for c, (off, n) in enumerate(zip(wl.pool_offsets, wl.chunk_lens))]
        chunks = [oracle.Chunk(off, n, 0) for off, n in zip(wl.pool_offsets, wl.chunk_lens)]
        pool = oracle.BlockPool(nb)
        plans, recs = [], []
        for req in mine.requests:
            plan, bt = pic.pic_build_block_table(ctx, [ids[c] for c, _ in req], 4096 // bs,
                                                 take_tokens=[t for _, t in req], k_nonleading=4)
            segs = oracle.compose(chunks, [c for c, _ in req], take=[t for _, t in req])
            want = pool.allocate(oracle.blocks_needed(4096, bs))
            assert bt[:len(want)].tolist() == want
            plans.append(plan)
            recs.append(oracle.recompute_positions(segs, 4, 0))
        indptr, idx = pic.pic_recompute_indices(plans)
        o_indptr, o_idx = oracle.recompute_csr(recs)
        assert np.array_equal(indptr, o_indptr) and np.array_equal(idx, o_idx)
        pic.pic_destroy(ctx)
        # the shards cover every request exactly once
        got = [None] * world
        dist.all_gather_object(got, list(range(lo, hi)))
        flat = [r for g in got for r in g]
        assert sorted(flat) == list(range(len(wl.requests))) and len(flat) == len(set(flat))
        # benchmark timing: the max over ranks
        assert max_over_ranks(1.5 + rank) == 1.5 + world - 1
        dist.barrier()
        dist.destroy_process_group()
    except BaseException as e:  # report to the parent, do not hang the group
        errq.put(f"rank {rank}: {type(e).__name__}: {e}")
        raise


def test_two_ranks_split_by_request():
    ctx = mp.get_context("spawn")
    errq = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, errq)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    alive = [p for p in procs if p.is_alive()]
    for p in alive:
        p.kill()
    errs = []
    while not errq.empty():
        errs.append(errq.get())
    assert not alive, "a rank did not finish"
    assert not errs, errs
    assert all(p.exitcode == 0 for p in procs)


def _tp_worker(rank, world, port, errq):
    try:
        import sys
        sys.path.insert(0, ROOT)
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle
        import workloads as W
        from harness import lib
        from position_independent_kv_stitch_gb300 import pic
        from position_independent_kv_stitch_gb300.sharding import shard_kv_heads
        lib()
        wl = W.tiny_gqa()
        m = wl.model
        lo, hi = shard_kv_heads(m.num_kv_heads, rank, world)
        mine = W.Model(**{**m.__dict__, "num_kv_heads": hi - lo})
        bs = m.block_size
        nb = -(-wl.request_tokens[0] // bs)
        ctx = pic.create_from_spec(pic.model_spec_from(mine), nb)
        ids = [pic.pic_register_chunk(ctx, W.chunk_key(wl.name, c), off, n)[0]
               for c, (off, n) in enumerate(zip(wl.pool_offsets, wl.chunk_lens))]
        req = wl.requests[0]
        plan, bt = pic.pic_build_block_table(ctx, [ids[c] for c, _ in req], nb, take_tokens=[t for _, t in req],
                                             k_nonleading=wl.k_nonleading, k_leading=wl.k_leading)
        indptr, idx = pic.pic_recompute_indices([plan])
        # the host plan does not depend on the heads: every rank has the same one
        got = [None] * world
        dist.all_gather_object(got, (bt.tolist(), indptr.tolist(), idx.tolist()))
        assert all(g == got[0] for g in got)
        pic.pic_destroy(ctx)
        # this rank's share of the stitched keys and values is the full
        # stitch's share: rotating a head needs no other head
        chunks = [oracle.Chunk(off, n, 0) for off, n in zip(wl.pool_offsets, wl.chunk_lens)]
        segs = oracle.compose(chunks, [c for c, _ in req], take=[t for _, t in req])
        table = bt[:nb].tolist()
        theta = oracle.model_inv_freq(m.rope_dim, m.rope_theta, m.llama3)
        kp = W.make_pool(wl, "k", "cpu").view(torch.int16).numpy().view(np.uint16)
        vp = W.make_pool(wl, "v", "cpu").view(torch.int16).numpy().view(np.uint16)
        full_k, full_v = oracle.stitch_paged(kp, vp, [segs], [table], nb, bs, theta, oracle.NEOX_HALF, 0, 128)
        part_k, part_v = oracle.stitch_paged(np.ascontiguousarray(kp[:, :, lo:hi]),
                                             np.ascontiguousarray(vp[:, :, lo:hi]), [segs], [table], nb, bs,
                                             theta, oracle.NEOX_HALF, 0, 128)
        assert np.array_equal(part_k, full_k[..., lo:hi, :], equal_nan=True)
        assert np.array_equal(part_v, full_v[..., lo:hi, :])
        heads = [None] * world
        dist.all_gather_object(heads, (lo, hi))
        assert sorted(heads) == [(r * (hi - lo), (r + 1) * (hi - lo)) for r in range(world)]
        dist.barrier()
        dist.destroy_process_group()
    except BaseException as e:  # report to the parent, do not hang the group
        errq.put(f"rank {rank}: {type(e).__name__}: {e}")
        raise


def test_two_ranks_split_kv_heads():
    """Tensor parallelism over KV heads (world size 2, gloo): the same plan on
    every rank, and each rank's stitched heads equal to its share of the
    full stitch."""
    ctx = mp.get_context("spawn")
    errq = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_tp_worker, args=(r, 2, port, errq)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    alive = [p for p in procs if p.is_alive()]
    for p in alive:
        p.kill()
    errs = []
    while not errq.empty():
        errs.append(errq.get())
    assert not alive, "a rank did not finish"
    assert not errs, errs
    assert all(p.exitcode == 0 for p in procs)


def test_shard_kv_heads_covers_every_head_once():
    from position_independent_kv_stitch_gb300.sharding import shard_kv_heads
    for h in (1, 2, 4, 8, 16):
        for world in (1, 2, 4, 8):
            if h % world:
                with pytest.raises(ValueError):
                    shard_kv_heads(h, 0, world)
                continue
            ranges = [shard_kv_heads(h, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == h
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            assert len({b - a for a, b in ranges}) == 1
    with pytest.raises(ValueError):
        shard_kv_heads(8, 4, 4)


def test_shard_requests_balanced_and_disjoint():
    from position_independent_kv_stitch_gb300.sharding import shard_requests
    for n in range(0, 20):
        for world in range(1, 9):
            ranges = [shard_requests(n, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [hi - lo for lo, hi in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_requests(4, 2, 2)
