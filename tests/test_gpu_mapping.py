"""GPU parity of virtual block mapping (EPIC runtime figure, steps 1-2):
mapped chunks rotate their keys in place, their values never move, copies
out of block-resident chunks and pool chunks land rotated, all in one launch,
under both kernel variants; results equal the oracle (keys within the
contract tolerance, everything else bit for bit)."""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from conftest import load_golden
from gpu_util import assert_k_close, bits, f64
from position_independent_kv_stitch_gb300 import pic

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pic.load(build_if_missing=True)


@pytest.fixture(params=["bulk", "regs"])
def variant(request, monkeypatch):
    monkeypatch.setenv("PIC_KERNEL", request.param)
    return request.param


def _model(kind, pairing, L, bs, H=2):
    if kind == "gqa":
        return W.Model("map", "gqa", L, H, 128, 128, 0, pairing, 5e5, bs, W.LLAMA3_SCALING)
    return W.Model("map", "mla", L, 1, 576, 64, 512, pairing, 1e4, bs)


def _run(m, nb, block_chunks, pool_chunks, requests, alias=True, k=(4, 0), seed=0, total=None):
    """block_chunks: {name: (blocks, n, base)}; pool_chunks: {name: (offset, n)};
    requests: list of name lists.  Returns everything needed to compare."""
    bs = m.block_size
    ctx = pic.create_from_spec(pic.model_spec_from(m), nb)
    shape = (m.num_layers, nb, bs) + tuple(m.row_shape)
    k_cache = torch.empty(shape, dtype=torch.bfloat16)
    W.fill_random_bf16(k_cache, seed, "map-k")
    v_cache = None
    if m.kind == "gqa":
        v_cache = torch.empty(shape, dtype=torch.bfloat16)
        W.fill_random_bf16(v_cache, seed, "map-v")
    P = max([o + n for o, n in pool_chunks.values()] + [16])
    k_pool = torch.empty((m.num_layers, P) + tuple(m.row_shape), dtype=torch.bfloat16)
    W.fill_random_bf16(k_pool, seed, "map-pk")
    v_pool = None
    if m.kind == "gqa":
        v_pool = torch.empty_like(k_pool)
        W.fill_random_bf16(v_pool, seed, "map-pv")
    ids, o_chunks = {}, {}
    opool = oracle.BlockPool(nb)
    for i, (name, (blks, n, base)) in enumerate(block_chunks.items()):
        ids[name] = pic.pic_register_chunk_blocks(ctx, W.chunk_key("mapb", i), blks, n, base)[0]
        o_chunks[name] = oracle.BlockChunk(tuple(blks), n, cur_pos=base)
        for b in blks:
            opool.free[b] = False
    for i, (name, (off, n)) in enumerate(pool_chunks.items()):
        ids[name] = pic.pic_register_chunk(ctx, W.chunk_key("mapp", i), off, n)[0]
        o_chunks[name] = oracle.Chunk(off, n, 0)
    plans, tables, o_plans = [], [], []
    mb = nb
    for r, names in enumerate(requests):
        kw = dict(total_tokens=total[r]) if total else {}
        plan, bt = pic.pic_build_block_table(ctx, [ids[n] for n in names], mb, alias=alias,
                                             k_nonleading=k[0], k_leading=k[1], **kw)
        segs, table, fresh, undo = oracle.map_request(o_chunks, names, bs, opool, r, alias=alias,
                                                      total_tokens=kw.get("total_tokens", 0))
        assert bt[:len(table)].tolist() == table
        plans.append(plan)
        tables.append(bt)
        o_plans.append((segs, table))
    dk, dv = k_cache.to(DEV), (v_cache.to(DEV) if v_cache is not None else None)
    dkp, dvp = k_pool.to(DEV), (v_pool.to(DEV) if v_pool is not None else None)
    d_bt = torch.from_numpy(np.stack(tables)).to(DEV)
    n_rec = len(pic.pic_recompute_indices(plans)[1])
    ridx = torch.full((max(1, n_rec),), -7, dtype=torch.int32, device=DEV)
    indptr = torch.empty(len(plans) + 1, dtype=torch.int32, device=DEV)
    ws = torch.empty(pic.pic_workspace_bytes(ctx, plans), dtype=torch.uint8, device=DEV)
    pic.pic_stitch(ctx, plans, dkp, dvp, dk, dv, d_bt, ridx, indptr, ws)
    assert pic.pic_query_device_status(ctx, ws) == 0
    # oracle: requests of one launch touch disjoint rows, so apply them one after another
    theta = oracle.model_inv_freq(m.rope_dim, m.rope_theta, m.llama3)
    pairing = oracle.NEOX_HALF if m.pairing == "neox" else oracle.INTERLEAVED
    kb = bits(k_cache)
    vb = bits(v_cache) if v_cache is not None else None
    want_k = oracle.bf16_bits_to_f64(kb)
    want_v = vb.copy() if vb is not None else None
    for segs, table in o_plans:
        k_o, v_o = oracle.apply_mapped(kb, vb, bits(k_pool), bits(v_pool) if v_pool is not None else None,
                                       segs, table, bs, theta, pairing, m.rope_offset, m.rope_dim)
        touched = np.zeros(want_k.shape[1:3], bool)
        for s in segs:
            for t in range(s.length):
                p = s.dst_pos + t
                touched[table[p // bs], p % bs] = True
        want_k[:, touched] = k_o[:, touched]
        if want_v is not None:
            want_v[:, touched] = v_o[:, touched]
    rec = [oracle.recompute_positions(
        [oracle.Segment(0, 0, s.length, s.dst_pos, s.delta) for s in segs], k[0], k[1]) for segs, _ in o_plans]
    return dict(ctx=ctx, plans=plans, k=dk, v=dv, want_k=want_k, want_v=want_v, ridx=ridx, indptr=indptr,
                rec=rec, n_rec=n_rec, k_before=kb, v_before=vb, args=(dkp, dvp, d_bt, ws), ids=ids,
                o_plans=o_plans)


def _check(res):
    got = f64(res["k"])
    assert_k_close(got, res["want_k"], "K")
    if res["want_v"] is not None:
        assert np.array_equal(bits(res["v"]), res["want_v"])
    indptr, idx = oracle.recompute_csr(res["rec"])
    assert res["indptr"].cpu().tolist() == indptr.tolist()
    assert res["ridx"].cpu().numpy()[:res["n_rec"]].tolist() == idx.tolist()


def test_epic_figure_zero_copy_on_gpu(variant):
    """System, DocB, DocA resident in blocks 102, 310..380, 204..250 and mapped
    into the request: keys rotate in place, values never move, no other row
    changes; the system block (delta 0) moves nothing but still reports its
    recompute positions."""
    g = load_golden("epic_virtual_block_mapping.json")
    ch = g["chunks"]
    blocks = {n: (d["blocks"] if "blocks" in d else list(range(d["blocks_range"][0], d["blocks_range"][1] + 1)))
              for n, d in ch.items()}
    m = _model("gqa", "neox", 2, 16)
    res = _run(m, 512, {n: (blocks[n], ch[n]["num_tokens"], ch[n]["base_pos"]) for n in ch}, {},
               [g["order"]], k=(4, 4), total=[g["expected_total_tokens"]])
    try:
        assert [pic.pic_plan_segment_mode(res["plans"][0], j) for j in range(3)] == [pic.PIC_SEG_MAPPED] * 3
        _check(res)
        # values untouched everywhere; keys changed only in the moved chunks' blocks
        assert np.array_equal(bits(res["v"]), res["v_before"])
        kb_after = bits(res["k"])
        moved = set(blocks["DocA"]) | set(blocks["DocB"])
        for b in range(512):
            same = np.array_equal(kb_after[:, b], res["k_before"][:, b])
            assert same == (b not in moved), b
        assert res["ridx"].cpu().numpy()[:res["n_rec"]].tolist()[:4] == [0, 1, 2, 3]
        # the plan's in-place rotations ran: a second stitch of it is refused
        with pytest.raises(pic.PicError) as e:
            pic.pic_stitch(res["ctx"], res["plans"], res["args"][0], res["args"][1], res["k"], res["v"],
                           res["args"][2], None, None, res["args"][3])
        assert e.value.status_name == "PIC_ERR_INVALID_ARG"
    finally:
        pic.pic_destroy(res["ctx"])


@pytest.mark.parametrize("kind,pairing", [("gqa", "neox"), ("gqa", "interleaved"), ("mla", "interleaved"),
                                          ("mla", "neox")])
def test_mixed_batch_copy_pool_copy_blocks_and_mapped(kind, pairing, variant):
    """Two requests in one launch: a mapped chunk, a block-resident chunk
    placed off a block boundary (copied out of its blocks), pool chunks, a
    chunk whose keys sit at a non-zero position."""
    m = _model(kind, pairing, 3, 16)
    block_chunks = {"A": ([7, 3, 11], 40, 300), "B": ([20, 21], 17, 0), "C": ([30], 16, 64)}
    pool_chunks = {"P": (0, 21), "Q": (21, 33)}
    requests = [["A", "P", "B", "Q"], ["C", "Q"]]
    res = _run(m, 64, block_chunks, pool_chunks, requests, seed=3)
    try:
        modes = [[pic.pic_plan_segment_mode(p, j) for j in range(len(r))] for p, r in zip(res["plans"], requests)]
        assert modes == [[pic.PIC_SEG_MAPPED, pic.PIC_SEG_COPY_POOL, pic.PIC_SEG_COPY_BLOCKS, pic.PIC_SEG_COPY_POOL],
                         [pic.PIC_SEG_MAPPED, pic.PIC_SEG_COPY_POOL]]
        _check(res)
    finally:
        pic.pic_destroy(res["ctx"])


def test_mapped_chunk_moves_again_by_the_difference():
    """A chunk mapped at 32, freed (stitched), mapped again at 0: the second
    shift is -32 and the keys end where the chunk's original keys would be
    rotated to 0 (two roundings)."""
    m = _model("gqa", "neox", 2, 16)
    res = _run(m, 32, {"A": ([5, 6], 32, 0), "S": ([9, 10], 32, 0)}, {}, [["S", "A"]])
    try:
        ctx = res["ctx"]
        _check(res)
        pic.pic_free_request(ctx, res["plans"][0])
        assert pic.pic_chunk_info(ctx, res["ids"]["A"])[2] == 32
        plan, bt = pic.pic_build_block_table(ctx, [res["ids"]["A"]], 4, alias=True)
        assert pic.pic_plan_segment(plan, 0)["delta"] == -32
        dkp, dvp, _, _ = res["args"]
        d_bt = torch.from_numpy(bt).to(DEV).view(1, -1)
        ws = torch.empty(pic.pic_workspace_bytes(ctx, [plan]), dtype=torch.uint8, device=DEV)
        pic.pic_stitch(ctx, [plan], dkp, dvp, res["k"], res["v"], d_bt, None, None, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0
        theta = oracle.model_inv_freq(128, 5e5, W.LLAMA3_SCALING)
        a, b = oracle.rope_pairs(128, oracle.NEOX_HALF)
        got = f64(res["k"])[:, [5, 6]]
        want = oracle.rotate(oracle.bf16_bits_to_f64(res["k_before"][:, [5, 6]]), 0, theta, oracle.NEOX_HALF)
        err = np.hypot(got[..., a] - want[..., a], got[..., b] - want[..., b])
        assert np.all(err <= 2.0 ** -7 * 1.01 * np.hypot(want[..., a], want[..., b]) + 1e-3)
        pic.pic_free_request(ctx, plan)
    finally:
        pic.pic_destroy(res["ctx"])


def test_llama_full_size_mapped_in_two_orders():
    """The mapped benchmark's launch at full size (Llama-3.1-8B RAG workload,
    32 layers, llama3-scaled theta): every chunk sits in its own cache blocks
    at position 0 and is mapped into the request (EPIC runtime figure, steps 1
    and 2: its blocks reused, its keys rotated in place, its values never
    moved).  Then the request is built again in a second order, so each chunk
    after the system prompt moves by the difference of its two positions.
    After each step, layers 0, 13 and 31 of every chunk are compared with
    the oracle's rotation of that layer's keys as they were before the step
    (one bf16 rounding per step); values, the request's own blocks, block
    tables and recompute lists must match bit for bit."""
    wl = W.llama31_8b_rag()
    m = wl.model
    bs = m.block_size
    theta = oracle.model_inv_freq(m.rope_dim, m.rope_theta, m.llama3)
    own_blocks = -(-wl.request_tokens[0] // bs)
    nblk = [-(-n // bs) for n in wl.chunk_lens]
    nb = own_blocks + sum(nblk)
    ctx = pic.create_from_spec(pic.model_spec_from(m), nb)
    try:
        k_pool = W.make_pool(wl, "k", device=DEV)
        v_pool = W.make_pool(wl, "v", device=DEV)
        shape = (m.num_layers, nb, bs) + tuple(m.row_shape)
        k_cache = torch.zeros(shape, dtype=torch.bfloat16, device=DEV)
        v_cache = torch.zeros(shape, dtype=torch.bfloat16, device=DEV)
        ids, blocks, first = [], [], own_blocks
        for c, (off, n) in enumerate(zip(wl.pool_offsets, wl.chunk_lens)):
            blks = list(range(first, first + nblk[c]))
            first += nblk[c]
            for j, b in enumerate(blks):
                t0, t1 = j * bs, min(n, (j + 1) * bs)
                k_cache[:, b, :t1 - t0] = k_pool[:, off + t0:off + t1]
                v_cache[:, b, :t1 - t0] = v_pool[:, off + t0:off + t1]
            ids.append(pic.pic_register_chunk_blocks(ctx, W.chunk_key(wl.name, c), blks, n, 0)[0])
            blocks.append(blks)
        v_before = v_cache.clone()
        head, rest = wl.requests[0][:1], list(wl.requests[0][1:])
        perm = W.Stream(1, "mapped/order/0").permutation(len(rest))
        orders = [wl.requests[0], head + [rest[i] for i in perm]]
        assert orders[0] != orders[1]
        layers = [0, 13, 31]
        pos_now = [0] * len(ids)  # where each chunk's keys sit
        for order in orders:
            plan, bt = pic.pic_build_block_table(ctx, [ids[c] for c, _ in order], own_blocks,
                                                 take_tokens=[t for _, t in order],
                                                 k_nonleading=wl.k_nonleading, k_leading=wl.k_leading, alias=True)
            # block-aligned chunks taken whole: all mapped, no fresh block
            assert bt.tolist() == [b for c, _ in order for b in blocks[c]]
            p, new_pos, rec = 0, {}, []
            for j, (c, n) in enumerate(order):
                assert pic.pic_plan_segment_mode(plan, j) == pic.PIC_SEG_MAPPED
                assert pic.pic_plan_segment(plan, j)["delta"] == p - pos_now[c]
                new_pos[c] = p
                rec += list(range(p, p + min(wl.k_leading if p == 0 else wl.k_nonleading, n)))
                p += n
            before = bits(k_cache[layers])
            ridx = torch.full((len(rec),), -7, dtype=torch.int32, device=DEV)
            indptr = torch.empty(2, dtype=torch.int32, device=DEV)
            ws = torch.empty(pic.pic_workspace_bytes(ctx, [plan]), dtype=torch.uint8, device=DEV)
            pic.pic_stitch(ctx, [plan], k_pool, v_pool, k_cache, v_cache, torch.from_numpy(bt).to(DEV).view(1, -1),
                           ridx, indptr, ws)
            assert pic.pic_query_device_status(ctx, ws) == 0
            assert ridx.cpu().tolist() == rec and indptr.cpu().tolist() == [0, len(rec)]
            after = k_cache[layers]
            for c, n in order:
                got = f64(after[:, blocks[c]].reshape(len(layers), -1, *m.row_shape)[:, :n])
                old = oracle.bf16_bits_to_f64(before[:, blocks[c]].reshape(len(layers), -1, *m.row_shape)[:, :n])
                assert_k_close(got, oracle.rotate(old, new_pos[c] - pos_now[c], theta, oracle.NEOX_HALF), f"K {c}")
            assert torch.equal(v_cache.view(torch.int16), v_before.view(torch.int16))
            assert not k_cache[:, :own_blocks].view(torch.int16).any()
            pic.pic_free_request(ctx, plan)
            for c in new_pos:
                pos_now[c] = new_pos[c]
                assert pic.pic_chunk_info(ctx, ids[c])[2] == new_pos[c]
    finally:
        pic.pic_destroy(ctx)
        torch.cuda.empty_cache()
