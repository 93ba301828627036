"""CPU tests of virtual block mapping through the C ABI's host side: block
tables, segment modes, shifts and the registry's exclusivity rules equal the
oracle's, step by step.  No kernel is launched."""

import numpy as np
import pytest

import oracle
import workloads as W
from conftest import load_golden
from harness import lib
from position_independent_kv_stitch_gb300 import pic
from position_independent_kv_stitch_gb300.pic import PicError

MODE = {"copy:pool": pic.PIC_SEG_COPY_POOL, "copy:cache": pic.PIC_SEG_COPY_BLOCKS, "alias:": pic.PIC_SEG_MAPPED}


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib()


def _ctx(nb, bs=16, L=2):
    return pic.pic_create(pic.PIC_KIND_GQA, L, 2, 64, 64, 0, pic.PIC_PAIRING_NEOX_HALF, bs, 1e4, nb)


def _check_plan(plan, bt, segs, table):
    info = pic.pic_plan_info(plan)
    assert info["num_segments"] == len(segs) and info["num_blocks"] == len(table)
    assert bt[:len(table)].tolist() == table
    for j, s in enumerate(segs):
        got = pic.pic_plan_segment(plan, j)
        assert (got["dst_pos"], got["delta"], got["num_tokens"]) == (s.dst_pos, s.delta, s.length)
        assert pic.pic_plan_segment_mode(plan, j) == MODE[f"{s.mode}:{s.src_kind}"]


def test_epic_figure_mapping_through_the_abi():
    g = load_golden("epic_virtual_block_mapping.json")
    ch = g["chunks"]
    blocks = {n: (d["blocks"] if "blocks" in d else list(range(d["blocks_range"][0], d["blocks_range"][1] + 1)))
              for n, d in ch.items()}
    ctx = _ctx(1024)
    try:
        ids = {n: pic.pic_register_chunk_blocks(ctx, W.chunk_key("fig", i), blocks[n], ch[n]["num_tokens"],
                                                ch[n]["base_pos"])[0] for i, n in enumerate(ch)}
        total = g["expected_total_tokens"]
        plan, bt = pic.pic_build_block_table(ctx, [ids[n] for n in g["order"]], 200, total_tokens=total, alias=True)
        want = blocks["System"] + blocks["DocB"] + blocks["DocA"]
        assert bt[:len(want)].tolist() == want and bt[len(want):len(want) + 2].tolist() == [0, 1]
        assert [pic.pic_plan_segment_mode(plan, j) for j in range(3)] == [pic.PIC_SEG_MAPPED] * 3
        assert [pic.pic_plan_segment(plan, j)["delta"] for j in range(3)] == g["expected_delta"]
        # the chunks now sit at their new positions; a second user is refused while mapped
        assert pic.pic_chunk_info(ctx, ids["DocA"])[2] == 1152
        with pytest.raises(PicError) as e:
            pic.pic_build_block_table(ctx, [ids["DocA"]], 100)
        assert e.value.status_name == "PIC_ERR_BUSY"
        with pytest.raises(PicError) as e:
            pic.pic_unregister_chunk(ctx, ids["DocB"])
        assert e.value.status_name == "PIC_ERR_BUSY"
        # freed without stitching: positions roll back
        pic.pic_free_request(ctx, plan)
        assert pic.pic_chunk_info(ctx, ids["DocA"])[2] == 0
    finally:
        pic.pic_destroy(ctx)


def test_mapping_sequences_match_oracle():
    """A sequence of requests mixing pool chunks and block-resident chunks,
    aligned and unaligned placements, repeats and live users, against the
    oracle's planner and registry state."""
    bs, nb = 4, 64
    ctx = _ctx(nb, bs)
    try:
        o_chunks = {}
        lib_id = {}
        pool = oracle.BlockPool(nb)
        # block-resident chunks (blocks chosen by hand) and pool chunks
        spec = {"X": ((3, 9), 8, 100), "Y": ((20, 21, 22), 10, 0), "Z": ((40,), 3, 7)}
        for i, (name, (blks, n, base)) in enumerate(spec.items()):
            lib_id[name] = pic.pic_register_chunk_blocks(ctx, W.chunk_key("seq", i), blks, n, base)[0]
            o_chunks[name] = oracle.BlockChunk(tuple(blks), n, cur_pos=base)
            for b in blks:
                pool.free[b] = False
        for i, (name, (off, n)) in enumerate({"P": (0, 5), "Q": (5, 6)}.items()):
            lib_id[name] = pic.pic_register_chunk(ctx, W.chunk_key("seqp", i), off, n)[0]
            o_chunks[name] = oracle.Chunk(off, n, 0)
        live = []
        steps = [(["X", "P", "Y"], True), (["Q", "Z"], True), (["P", "Q"], False), ("free", 0),
                 (["Y", "X"], True), (["Z", "Z"], True), ("free", 1), (["X"], False), ("free", 0), ("free", 0),
                 (["Z", "P", "X", "Y"], True)]
        for k, step in enumerate(steps):
            if step[0] == "free":
                plan, segs, fresh, undo = live.pop(step[1])
                pic.pic_free_request(ctx, plan)
                oracle.release_request(o_chunks, segs, fresh, undo, pool, applied=False)
                continue
            names, alias = step
            try:
                segs, table, fresh, undo = oracle.map_request(o_chunks, names, bs, pool, f"r{k}", alias=alias)
            except oracle.BusyError:
                with pytest.raises(PicError) as e:
                    pic.pic_build_block_table(ctx, [lib_id[n] for n in names], 32, alias=alias)
                assert e.value.status_name == "PIC_ERR_BUSY"
                continue
            plan, bt = pic.pic_build_block_table(ctx, [lib_id[n] for n in names], 32, alias=alias)
            _check_plan(plan, bt, segs, table)
            live.append((plan, segs, fresh, undo))
            for name in spec:
                assert pic.pic_chunk_info(ctx, lib_id[name])[2] == o_chunks[name].cur_pos
        assert any(s.mode == "alias" for _, ss, _, _ in live for s in ss)
    finally:
        pic.pic_destroy(ctx)


def test_register_blocks_validation():
    ctx = _ctx(8, 4)
    try:
        pic.pic_register_chunk_blocks(ctx, W.chunk_key("v", 0), [1, 2], 8)
        with pytest.raises(PicError) as e:        # block 2 already taken
            pic.pic_register_chunk_blocks(ctx, W.chunk_key("v", 1), [2], 3)
        assert e.value.status_name == "PIC_ERR_RANGE"
        with pytest.raises(PicError) as e:        # outside the cache
            pic.pic_register_chunk_blocks(ctx, W.chunk_key("v", 2), [8], 3)
        assert e.value.status_name == "PIC_ERR_RANGE"
        with pytest.raises(PicError) as e:        # listed twice
            pic.pic_register_chunk_blocks(ctx, W.chunk_key("v", 3), [5, 5], 6)
        assert e.value.status_name == "PIC_ERR_INVALID_ARG"
        # more blocks than the cache holds (9 > 8; and 2^31 - 1 tokens, whose
        # block count once overflowed int32): refused before blocks[] is read
        for n in (33, 2**31 - 1):
            with pytest.raises(PicError) as e:
                pic.pic_register_chunk_blocks(ctx, W.chunk_key("v", 4), [6], n)
            assert e.value.status_name == "PIC_ERR_RANGE"
        # same key, same blocks: the existing id
        assert pic.pic_register_chunk_blocks(ctx, W.chunk_key("v", 0), [1, 2], 8) == (0, False)
        # the chunk's blocks are out of the allocator: a 6-block request gets 0, 3..7
        plan, bt = pic.pic_build_block_table(ctx, [], 6, total_tokens=24)
        assert bt.tolist() == [0, 3, 4, 5, 6, 7]
        pic.pic_free_request(ctx, plan)
        pic.pic_unregister_chunk(ctx, 0)          # blocks come back
        plan, bt = pic.pic_build_block_table(ctx, [], 8, total_tokens=32)
        assert bt.tolist() == list(range(8))
    finally:
        pic.pic_destroy(ctx)
