"""CPU tests of the C ABI: the library loads and exports every declared symbol,
and its host logic (registry, composer, block allocator, recompute list,
argument validation) matches the oracle bit for bit.  No kernel is launched."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads as W
from harness import (blocks_for, create_ctx, lib, lib_plan, lib_register, max_blocks_for,
                     oracle_plan)
from position_independent_kv_stitch_gb300 import pic
from position_independent_kv_stitch_gb300.pic import PicError

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    lib()


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pic_[a-z_0-9]+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    declared = _declared_functions()
    assert "pic_stitch" in declared and "pic_rerotate_inplace" in declared
    so = ctypes.CDLL(pic.lib_path())
    missing = [n for n in sorted(declared) if not hasattr(so, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert pic.pic_abi_version() == 2


def test_binding_covers_every_declared_function():
    assert _declared_functions() <= set(pic._SIGNATURES)


@pytest.mark.parametrize("name", ["tiny_gqa", "llama31_8b_rag", "qwen3_8b_batch", "deepseek_v3_mla",
                                  "serving_stress"])
def test_plans_tables_and_recompute_match_oracle(name):
    wl = W.WORKLOADS[name]()
    nb = blocks_for(wl) + 7
    ctx = create_ctx(wl, nb)
    try:
        ids = lib_register(ctx, wl)
        assert ids == list(range(len(wl.chunk_lens)))
        plans, tables = lib_plan(ctx, wl, ids)
        o_segs, o_tables, o_rec = oracle_plan(wl, nb)
        mb = max_blocks_for(wl)
        for r, plan in enumerate(plans):
            info = pic.pic_plan_info(plan)
            assert info["num_segments"] == len(o_segs[r])
            for j, s in enumerate(o_segs[r]):
                got = pic.pic_plan_segment(plan, j)
                assert (got["src_tok"], got["num_tokens"], got["dst_pos"], got["delta"]) == \
                       (s.src_tok, s.length, s.dst_pos, s.delta)
            want = np.full(mb, -1, np.int32)
            want[:len(o_tables[r])] = o_tables[r]
            np.testing.assert_array_equal(tables[r], want)
        indptr, idx = pic.pic_recompute_indices(plans)
        o_indptr, o_idx = oracle.recompute_csr(o_rec)
        np.testing.assert_array_equal(indptr, o_indptr)
        np.testing.assert_array_equal(idx, o_idx)
    finally:
        pic.pic_destroy(ctx)


def test_free_and_reallocate_matches_oracle_pool():
    wl = W.tiny_gqa()
    ctx = create_ctx(wl, 300)
    pool = oracle.BlockPool(300)
    try:
        ids = lib_register(ctx, wl)
        live = []
        seq = [(0, 2, 3), (1,), (0, 1), (4, 3, 2, 1), (2,), (0,)]
        for step, chosen in enumerate(seq):
            plan, bt = pic.pic_build_block_table(ctx, [ids[c] for c in chosen], 80)
            total = sum(wl.chunk_lens[c] for c in chosen)
            want = pool.allocate(oracle.blocks_needed(total, 16))
            assert bt[:len(want)].tolist() == want and np.all(bt[len(want):] == -1)
            live.append((plan, want))
            if step % 2 == 1:  # free the oldest live request
                p, blocks = live.pop(0)
                pic.pic_free_request(ctx, p)
                pool.release(blocks)
    finally:
        pic.pic_destroy(ctx)


def _gqa_ctx(nb=64, **kw):
    args = dict(kind=pic.PIC_KIND_GQA, num_layers=2, num_kv_heads=2, head_dim=128, rope_dim=128,
                rope_offset=0, pairing=pic.PIC_PAIRING_NEOX_HALF, block_size=16, rope_theta=1e4,
                num_cache_blocks=nb)
    args.update(kw)
    return pic.pic_create(**args)


def test_create_validation():
    with pytest.raises(PicError) as e:
        _gqa_ctx(head_dim=96, rope_dim=96)
    assert e.value.status_name == "PIC_ERR_UNSUPPORTED"
    with pytest.raises(PicError) as e:
        _gqa_ctx(rope_dim=64)
    assert e.value.status_name == "PIC_ERR_UNSUPPORTED"
    with pytest.raises(PicError) as e:
        _gqa_ctx(pairing=7)
    assert e.value.status_name == "PIC_ERR_INVALID_ARG"
    with pytest.raises(PicError) as e:
        _gqa_ctx(block_size=0)
    assert e.value.status_name == "PIC_ERR_INVALID_ARG"
    with pytest.raises(PicError) as e:
        pic.pic_create(pic.PIC_KIND_MLA, 2, 1, 512, 64, 448, 1, 16, 1e4, 8)
    assert e.value.status_name == "PIC_ERR_UNSUPPORTED"
    with pytest.raises(PicError):
        _gqa_ctx(rope_theta=1.0)
    assert "rope_theta" in pic.pic_last_error(None)


def test_registry_semantics():
    ctx = _gqa_ctx()
    try:
        k1, k2 = W.chunk_key("r", 1), W.chunk_key("r", 2)
        assert pic.pic_register_chunk(ctx, k1, 0, 10) == (0, True)
        assert pic.pic_register_chunk(ctx, k1, 999, 10) == (0, False)  # same key, same length
        assert pic.pic_chunk_info(ctx, 0) == (0, 10, 0)                 # first offset kept
        with pytest.raises(PicError) as e:
            pic.pic_register_chunk(ctx, k1, 0, 11)
        assert e.value.status_name == "PIC_ERR_KEY_CONFLICT"
        with pytest.raises(PicError) as e:
            pic.pic_register_chunk(ctx, k1, 0, 10, base_pos=5)
        assert e.value.status_name == "PIC_ERR_KEY_CONFLICT"
        assert pic.pic_register_chunk(ctx, k2, 10, 7, base_pos=3) == (1, True)
        assert pic.pic_lookup_chunk(ctx, k2) == 1
        pic.pic_unregister_chunk(ctx, 1)
        with pytest.raises(PicError) as e:
            pic.pic_lookup_chunk(ctx, k2)
        assert e.value.status_name == "PIC_ERR_UNKNOWN_CHUNK"
        with pytest.raises(PicError) as e:
            pic.pic_build_block_table(ctx, [1], 4)
        assert e.value.status_name == "PIC_ERR_UNKNOWN_CHUNK"
        # the id is not reused
        assert pic.pic_register_chunk(ctx, k2, 10, 7, base_pos=3) == (2, True)
        with pytest.raises(PicError) as e:
            pic.pic_register_chunk(ctx, W.chunk_key("r", 3), -1, 7)
        assert e.value.status_name == "PIC_ERR_RANGE"
    finally:
        pic.pic_destroy(ctx)


def test_plan_errors_leave_allocator_untouched():
    ctx = _gqa_ctx(nb=4)
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("e", 0), 0, 40)
        pic.pic_register_chunk(ctx, W.chunk_key("e", 1), 40, 40)
        with pytest.raises(PicError) as e:
            pic.pic_build_block_table(ctx, [0, 1], 8)           # needs 5 blocks, 4 exist
        assert e.value.status_name == "PIC_ERR_OUT_OF_BLOCKS"
        with pytest.raises(PicError) as e:
            pic.pic_build_block_table(ctx, [0, 1], 4)           # table too short
        assert e.value.status_name == "PIC_ERR_CAPACITY"
        with pytest.raises(PicError) as e:
            pic.pic_build_block_table(ctx, [0, 1], 8, dst_pos=[0, 30])   # overlap
        assert e.value.status_name == "PIC_ERR_RANGE"
        with pytest.raises(PicError) as e:
            pic.pic_build_block_table(ctx, [0], 8, take_tokens=[41])
        assert e.value.status_name == "PIC_ERR_RANGE"
        with pytest.raises(PicError) as e:
            pic.pic_build_block_table(ctx, [0], 8, total_tokens=39)
        assert e.value.status_name == "PIC_ERR_RANGE"
        with pytest.raises(PicError) as e:
            pic.pic_build_block_table(ctx, [0], 2 ** 20 + 8, start_pos=2 ** 24)  # |delta| >= 2^24
        assert e.value.status_name == "PIC_ERR_RANGE"
        # nothing leaked: all 4 blocks still allocatable
        plan, bt = pic.pic_build_block_table(ctx, [0, 1], 8, take_tokens=[40, 24])
        assert bt.tolist() == [0, 1, 2, 3, -1, -1, -1, -1]
        pic.pic_free_request(ctx, plan)
        with pytest.raises(PicError):
            pic.pic_free_request(ctx, plan)                     # double free is refused
    finally:
        pic.pic_destroy(ctx)


def test_explicit_positions_total_tokens_and_recompute():
    """EPIC client request: chunks at explicit offsets 128 and 4224, inline tokens around them."""
    ctx = _gqa_ctx(nb=400)
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("c", 0), 0, 1024)
        pic.pic_register_chunk(ctx, W.chunk_key("c", 1), 1024, 1024)
        plan, bt = pic.pic_build_block_table(ctx, [0, 1], 400, dst_pos=[128, 4224], total_tokens=5300,
                                             k_nonleading=4)
        info = pic.pic_plan_info(plan)
        assert info["total_tokens"] == 5300 and info["num_blocks"] == 332 and info["num_recompute"] == 8
        assert pic.pic_plan_segment(plan, 1)["delta"] == 4224
        indptr, idx = pic.pic_recompute_indices([plan])
        assert idx.tolist() == [128, 129, 130, 131, 4224, 4225, 4226, 4227] and indptr.tolist() == [0, 8]
    finally:
        pic.pic_destroy(ctx)


def test_recompute_list_beyond_int32_offsets_is_refused():
    # One request of 2^30 + 1 tokens whose chunk (at position 1) is all
    # recompute tokens; the same plan listed three times holds 3 * 2^30
    # entries, more than the int32 CSR offsets address.
    bs, n = 256, 2**30
    nb = n // bs + 1
    ctx = pic.pic_create(pic.PIC_KIND_GQA, 1, 1, 64, 64, 0, pic.PIC_PAIRING_NEOX_HALF, bs, 1e4, nb)
    try:
        cid, _ = pic.pic_register_chunk(ctx, W.chunk_key("big", 0), 0, n)
        plan, _ = pic.pic_build_block_table(ctx, [cid], nb, start_pos=1, k_nonleading=n)
        assert pic.pic_plan_info(plan)["num_recompute"] == n
        count = ctypes.c_int64()
        one = pic._plan_array([plan])
        assert pic.load().pic_recompute_indices(one, 1, None, None, 0, ctypes.byref(count)) == 0
        assert count.value == n
        with pytest.raises(PicError) as e:
            pic.pic_recompute_indices([plan] * 3)
        assert e.value.status_name == "PIC_ERR_RANGE"
        # the stitch's device CSR has the same limit; refused on the host
        # (fake, aligned pointers that never reach a launch)
        good = ctypes.c_void_p(0x10000)
        st = pic.load().pic_stitch(ctx, pic._plan_array([plan] * 3), 3, good, good, 0, good, good, 0, good, nb,
                                   good, good, 1 << 40, good, 1 << 40, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_RANGE"
        pic.pic_free_request(ctx, plan)
    finally:
        pic.pic_destroy(ctx)


def test_stitch_argument_checks_need_no_gpu():
    """Validation fails before anything is enqueued (no GPU needed to see it).
    Every call here must fail a host check: the pointers are fake."""
    ctx = _gqa_ctx(nb=8)
    L = pic.load()
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("s", 0), 0, 20)
        # start_pos 5: the chunk is non-leading, so the plan has 4 recompute entries
        plan, _ = pic.pic_build_block_table(ctx, [0], 4, start_pos=5, k_nonleading=4)
        assert pic.pic_plan_info(plan)["num_recompute"] == 4
        arr = pic._plan_array([plan])
        good = ctypes.c_void_p(0x10000)
        odd = ctypes.c_void_p(0x10008)
        ls = 8 * 16 * 512
        # GQA without values
        st = L.pic_stitch(ctx, arr, 1, good, None, ls, good, None, ls, good, 4, None, None, 0, good, 1 << 20, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_INVALID_ARG"
        # misaligned cache
        st = L.pic_stitch(ctx, arr, 1, good, good, ls, odd, good, ls, good, 4, None, None, 0, good, 1 << 20, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_ALIGNMENT"
        # block-table rows too short for the plan (needs 2 blocks)
        st = L.pic_stitch(ctx, arr, 1, good, good, ls, good, good, ls, good, 1, None, None, 0, good, 1 << 20, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_CAPACITY"
        # recompute capacity too small
        st = L.pic_stitch(ctx, arr, 1, good, good, ls, good, good, ls, good, 4, good, good, 0, good, 1 << 20, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_CAPACITY"
        # workspace too small
        need = pic.pic_workspace_bytes(ctx, [plan])
        assert need > 0 and need % 256 == 0
        st = L.pic_stitch(ctx, arr, 1, good, good, ls, good, good, ls, good, 4, None, None, 0, good, need - 1, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_CAPACITY"
        # cache layer stride smaller than the cache
        st = L.pic_stitch(ctx, arr, 1, good, good, ls, good, good, 16, good, 4, None, None, 0, good, need, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_RANGE"
        # a plan from another context
        ctx2 = _gqa_ctx(nb=8)
        st = L.pic_stitch(ctx2, arr, 1, good, good, ls, good, good, ls, good, 4, None, None, 0, good, need, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_INVALID_ARG"
        pic.pic_destroy(ctx2)
        # in-place: delta beyond range, req beyond tables
        segs = pic._shift_array([(0, 0, 4, 1 << 24)])
        st = L.pic_rerotate_inplace(ctx, good, ls, good, 1, 4, segs, 1, good, 1 << 20, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_RANGE"
        segs = pic._shift_array([(1, 0, 4, 5)])
        st = L.pic_rerotate_inplace(ctx, good, ls, good, 1, 4, segs, 1, good, 1 << 20, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_RANGE"
        segs = pic._shift_array([(0, 60, 5, 5)])  # ends past 4 blocks of 16
        st = L.pic_rerotate_inplace(ctx, good, ls, good, 1, 4, segs, 1, good, 1 << 20, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_RANGE"
        # within a (claimed) 2^27-block table, but ending past int32 positions
        segs = pic._shift_array([(0, 2**31 - 8, 16, 5)])
        st = L.pic_rerotate_inplace(ctx, good, ls, good, 1, 2**27, segs, 1, good, 1 << 20, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_RANGE"
    finally:
        pic.pic_destroy(ctx)


def test_pool_read_rows_count_repeats_once():
    """pic_pool_read_rows against the plans' own segments: every pool row a
    segment reads counts once in the distinct total however many segments
    read it; block-resident chunks read no pool rows."""
    ctx = _gqa_ctx(nb=64)
    try:
        lens = [20, 7, 33, 16]
        offs = [0, 20, 27, 60]
        ids = [pic.pic_register_chunk(ctx, W.chunk_key("rows", c), offs[c], lens[c])[0] for c in range(4)]
        bid = pic.pic_register_chunk_blocks(ctx, W.chunk_key("rows", 9), [60, 61], 20)[0]
        plans = [pic.pic_build_block_table(ctx, [ids[0], ids[2], ids[0], bid], 8)[0],
                 pic.pic_build_block_table(ctx, [ids[2], ids[3]], 8, take_tokens=[10, 16])[0],
                 pic.pic_build_block_table(ctx, [bid], 4)[0]]
        rows, read = set(), 0
        for plan in plans:
            for j in range(pic.pic_plan_info(plan)["num_segments"]):
                sg = pic.pic_plan_segment(plan, j)
                if sg["src_tok"] >= 0:
                    rows |= set(range(sg["src_tok"], sg["src_tok"] + sg["num_tokens"]))
                    read += sg["num_tokens"]
        assert (len(rows), read) == (20 + 33 + 16, 20 + 33 + 20 + 10 + 16)
        assert pic.pic_pool_read_rows(ctx, plans) == (len(rows), read)
        assert pic.pic_pool_read_rows(ctx, plans[2:]) == (0, 0)
        assert pic.pic_pool_read_rows(ctx, []) == (0, 0)
        # rows an earlier group staged are left out: plan 1 reads rows 27-36
        # (of chunk 2, which plan 0 reads whole) and 60-75
        assert pic.pic_pool_read_rows(ctx, plans[1:2], staged_plans=plans[:1]) == (16, 26)
        assert pic.pic_pool_read_rows(ctx, plans[:1], staged_plans=plans[1:2]) == (20 + 33 - 10, 73)
        assert pic.pic_pool_read_rows(ctx, plans, staged_plans=plans) == (0, read)
        # the groups' distinct rows add up to the batch's
        assert (pic.pic_pool_read_rows(ctx, plans[:1])[0] + pic.pic_pool_read_rows(ctx, plans[1:], plans[:1])[0]
                == len(rows))
        ctx2 = _gqa_ctx(nb=8)
        with pytest.raises(PicError) as e:
            pic.pic_pool_read_rows(ctx2, plans[:1])
        assert e.value.status_name == "PIC_ERR_INVALID_ARG"
        pic.pic_destroy(ctx2)
    finally:
        pic.pic_destroy(ctx)


def test_stage_pool_argument_checks_need_no_gpu():
    """pic_stage_pool refuses bad arguments before any CUDA call (fake,
    aligned pointers that never reach a copy)."""
    ctx = _gqa_ctx(nb=8)
    L = pic.load()
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("st", 0), 100, 20)
        plan, _ = pic.pic_build_block_table(ctx, [0], 4)
        arr = pic._plan_array([plan])
        good, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008)
        ls = 120 * 512  # rows 100-119 of 512 bytes (2 heads x 128 dims x bf16) fit
        n = ctypes.c_int64(-1)
        # GQA without value pools
        st = L.pic_stage_pool(ctx, arr, 1, None, 0, good, None, ls, good, None, ls, ctypes.byref(n), None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_INVALID_ARG"
        # misaligned device pool, then a misaligned stride
        st = L.pic_stage_pool(ctx, arr, 1, None, 0, good, good, ls, good, odd, ls, ctypes.byref(n), None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_ALIGNMENT"
        st = L.pic_stage_pool(ctx, arr, 1, None, 0, good, good, ls + 8, good, good, ls, ctypes.byref(n), None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_ALIGNMENT"
        # a layer stride that does not reach row 119 (two layers)
        st = L.pic_stage_pool(ctx, arr, 1, None, 0, good, good, ls, good, good, ls - 512, ctypes.byref(n), None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_RANGE"
        # null context, a bad plan list
        st = L.pic_stage_pool(None, arr, 1, None, 0, good, good, ls, good, good, ls, ctypes.byref(n), None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_INVALID_ARG"
        st = L.pic_stage_pool(ctx, None, 1, None, 0, good, good, ls, good, good, ls, ctypes.byref(n), None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_INVALID_ARG"
        assert n.value == -1
    finally:
        pic.pic_destroy(ctx)
    mla = pic.pic_create(kind=pic.PIC_KIND_MLA, num_layers=1, num_kv_heads=1, head_dim=576, rope_dim=64,
                         rope_offset=512, pairing=pic.PIC_PAIRING_INTERLEAVED, block_size=16, rope_theta=1e4,
                         num_cache_blocks=8)
    try:
        pic.pic_register_chunk(mla, W.chunk_key("st", 1), 0, 20)
        plan, _ = pic.pic_build_block_table(mla, [0], 4)
        arr = pic._plan_array([plan])
        good = ctypes.c_void_p(0x10000)
        # MLA rows have no value pools
        st = L.pic_stage_pool(mla, arr, 1, None, 0, good, good, 0, good, None, 0, None, None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_INVALID_ARG"
    finally:
        pic.pic_destroy(mla)


def test_staged_stitch_workspace_and_argument_checks_need_no_gpu():
    """pic_stitch_staged's workspace is one stitch image per request group
    (one group: pic_stitch's own size); bad arguments are refused before any
    CUDA call (fake, aligned pointers)."""
    ctx = _gqa_ctx(nb=32)
    L = pic.load()
    try:
        for c, n in enumerate([20, 7, 33]):
            pic.pic_register_chunk(ctx, W.chunk_key("sg", c), [0, 20, 27][c], n)
        plans = [pic.pic_build_block_table(ctx, ids, 6, k_nonleading=4)[0] for ids in ([0, 2], [1, 0], [2], [1])]
        one = pic.pic_stitch_staged_workspace_bytes(ctx, plans, 1)
        assert one == pic.pic_workspace_bytes(ctx, plans)
        per = [pic.pic_workspace_bytes(ctx, [p]) for p in plans]
        assert pic.pic_stitch_staged_workspace_bytes(ctx, plans, 4) == sum(per)
        assert pic.pic_stitch_staged_workspace_bytes(ctx, plans, 99) == sum(per)   # clamped to 4 groups
        assert pic.pic_stitch_staged_workspace_bytes(ctx, plans, 2) == (pic.pic_workspace_bytes(ctx, plans[:2])
                                                                         + pic.pic_workspace_bytes(ctx, plans[2:]))
        assert pic.pic_stitch_staged_workspace_bytes(ctx, plans, 0) == 0
        arr = pic._plan_array(plans)
        good = ctypes.c_void_p(0x10000)
        pls = 60 * 512
        cls = 32 * 16 * 512

        def call(n_groups, ws_bytes, cache=good, pool_ls=pls):
            return pic.STATUS_NAMES[L.pic_stitch_staged(ctx, arr, 4, n_groups, good, good, pool_ls, good, good, pool_ls,
                                                        cache, good, cls, good, 6, None, None, 0, good, ws_bytes,
                                                        None, None)]
        assert call(0, 1 << 20) == "PIC_ERR_INVALID_ARG"
        assert call(2, pic.pic_stitch_staged_workspace_bytes(ctx, plans, 2) - 1) == "PIC_ERR_CAPACITY"
        assert call(2, 1 << 20, cache=ctypes.c_void_p(0x10008)) == "PIC_ERR_ALIGNMENT"
        assert call(2, 1 << 20, pool_ls=59 * 512) == "PIC_ERR_RANGE"   # rows up to 59 are read
    finally:
        pic.pic_destroy(ctx)


def test_attend_argument_checks_need_no_gpu():
    """pic_attend_decode refuses bad arguments before any CUDA call (fake,
    aligned pointers that never reach a launch)."""
    ctx = _gqa_ctx(nb=8)  # 2 layers, 2 KV heads of 128 dims
    L = pic.load()
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("a", 0), 0, 20)
        plan, _ = pic.pic_build_block_table(ctx, [0], 4)
        arr = pic._plan_array([plan])
        g, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008)
        ls = 8 * 16 * 512

        def call(source=pic.PIC_ATTEND_FUSED, q=g, hq=4, lb=0, nl=2, plans=arr, n=1):
            st = L.pic_attend_decode(ctx, plans, n, source, q, hq, 0.1, 0.0, g, g, ls, g, g, ls, lb, nl,
                                     g, None, g, 1 << 20, None)
            return pic.STATUS_NAMES[st]

        assert call(source=7) == "PIC_ERR_INVALID_ARG"
        assert call(hq=6) == "PIC_ERR_UNSUPPORTED"          # 3 query heads per KV head
        assert call(hq=3) == "PIC_ERR_INVALID_ARG"          # not a multiple of the KV heads
        assert call(lb=1, nl=2) == "PIC_ERR_RANGE"
        assert call(lb=2**31 - 1, nl=1) == "PIC_ERR_RANGE"  # the sum once wrapped past int32
        assert call(nl=0) == "PIC_ERR_RANGE"
        assert call(q=None) == "PIC_ERR_INVALID_ARG"
        assert call(q=odd) == "PIC_ERR_ALIGNMENT"
        assert call(n=0) == "PIC_ERR_INVALID_ARG"
        empty, _ = pic.pic_build_block_table(ctx, [], 4)
        assert call(plans=pic._plan_array([empty])) == "PIC_ERR_RANGE"  # no context to attend
        pic.pic_free_request(ctx, empty)
        pic.pic_free_request(ctx, plan)
    finally:
        pic.pic_destroy(ctx)


def test_workspace_sizes_grow_with_runs():
    ctx = _gqa_ctx(nb=64)
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("w", 0), 0, 16)
        pic.pic_register_chunk(ctx, W.chunk_key("w", 1), 16, 17)
        p1, _ = pic.pic_build_block_table(ctx, [0], 8)
        p2, _ = pic.pic_build_block_table(ctx, [0, 1, 0, 1], 8, start_pos=3)
        assert pic.pic_workspace_bytes(ctx, [p2]) >= pic.pic_workspace_bytes(ctx, [p1])
        assert pic.pic_rerotate_workspace_bytes(ctx, [(0, 3, 40, 7)]) > pic.pic_rerotate_workspace_bytes(ctx, [(0, 3, 40, 0)])
    finally:
        pic.pic_destroy(ctx)


def test_debug_stall_hook_checks_its_context():
    L = pic.load()
    assert pic.STATUS_NAMES[L.pic_debug_stall_next_launch(None, 2, 1000)] == "PIC_ERR_INVALID_ARG"
    ctx = _gqa_ctx(nb=8)
    try:
        pic.pic_debug_stall_next_launch(ctx, 2, 1000)
        pic.pic_debug_stall_next_launch(ctx, -1)
    finally:
        pic.pic_destroy(ctx)


def test_kernel_variant_of_decode_attention(monkeypatch):
    """Mode 2 reports the decode-attention kernel chosen at pic_create: tcgen05
    for MLA models unless PIC_ATTEND_KERNEL=mma, warp-level mma for GQA."""
    mla = W.deepseek_v3_mla(context_tokens=256, num_layers=1).model
    monkeypatch.delenv("PIC_ATTEND_KERNEL", raising=False)
    ctx = pic.create_from_spec(pic.model_spec_from(mla), 32)
    try:
        assert pic.pic_kernel_variant(ctx, 2) == pic.PIC_VARIANT_TENSOR_CORE_TMEM
        assert pic.pic_kernel_variant(ctx, 3) == -1
    finally:
        pic.pic_destroy(ctx)
    monkeypatch.setenv("PIC_ATTEND_KERNEL", "mma")
    ctx = pic.create_from_spec(pic.model_spec_from(mla), 32)
    try:
        assert pic.pic_kernel_variant(ctx, 2) == pic.PIC_VARIANT_WARP_MMA
    finally:
        pic.pic_destroy(ctx)
    monkeypatch.delenv("PIC_ATTEND_KERNEL")
    ctx = _gqa_ctx(nb=8)
    try:
        assert pic.pic_kernel_variant(ctx, 2) == pic.PIC_VARIANT_WARP_MMA
    finally:
        pic.pic_destroy(ctx)
