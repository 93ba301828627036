"""Pools and caches in pinned host memory: the kernels stream them over the
host link directly.  Results must equal the device-memory path bit for bit
and match the oracle; pageable host memory is refused before any launch."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import Stitched, assert_k_close, bits, f64, oracle_side, pairing_of, theta_of
from position_independent_kv_stitch_gb300 import pic

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pic.load(build_if_missing=True)


def _pinned_like(t):
    return torch.empty(t.shape, dtype=t.dtype).pin_memory()


@pytest.mark.parametrize("name", ["tiny_gqa", "mla_small"])
def test_host_pool_and_cache_match_device_path_and_oracle(name):
    if name == "tiny_gqa":
        wl = W.tiny_gqa()
    else:
        base = W.deepseek_v3_mla(context_tokens=1500, num_layers=2)
        wl = W.Workload("mla-host", base.model, base.chunk_lens, base.requests, 0, 32)
    dev = Stitched(wl, pool_device="cpu").run()
    try:
        hk = dev.k_pool.cpu().pin_memory()
        hv = dev.v_pool.cpu().pin_memory() if dev.v_pool is not None else None
        hkc = _pinned_like(dev.k_cache)
        hkc.view(torch.int16).fill_(-1)
        hvc = None
        if dev.v_cache is not None:
            hvc = _pinned_like(dev.v_cache)
            hvc.view(torch.int16).fill_(-1)
        ws = torch.empty_like(dev.ws)
        ridx = torch.empty_like(dev.ridx)
        indptr = torch.empty_like(dev.indptr)
        pic.pic_stitch(dev.ctx, dev.plans, hk, hv, hkc, hvc, dev.d_bt, ridx, indptr, ws)
        assert pic.pic_query_device_status(dev.ctx, ws) == 0
        torch.cuda.synchronize()
        assert np.array_equal(bits(hkc), bits(dev.k_cache))
        if hvc is not None:
            assert np.array_equal(bits(hvc), bits(dev.v_cache))
        assert torch.equal(ridx, dev.ridx) and torch.equal(indptr, dev.indptr)
        segs, tables, _ = oracle_side(wl, dev.nb)
        m = wl.model
        want_k, _ = oracle.stitch_paged(bits(hk), None, segs, tables, dev.nb, dev.bs, theta_of(m),
                                        pairing_of(m), m.rope_offset, m.rope_dim)
        assert_k_close(f64(hkc), want_k, "host K")
    finally:
        dev.close()


@pytest.mark.parametrize("kind", ["gqa", "mla"])
def test_staged_pool_copies_each_row_read_once_and_stitches_the_same(kind):
    """pic_stage_pool from a pinned host pool into a zeroed device pool: the
    rows the plans read arrive bit for bit, every other row stays zero, and
    the stitch from the staged pool equals the stitch from the full device
    pool bit for bit (the same kernel on the same rows), which the oracle
    checks.  Chunks 1 and 4 are never read; chunk 2 is read three times, in
    two requests; chunk 3 in part.  The rows are staged in two calls, the
    second skipping the rows of the first request."""
    lens = [40, 17, 100, 33, 9, 64]
    reqs = [[(2, 100), (0, 40), (3, 20), (2, 100)], [(5, 64), (2, 50), (0, 40)]]
    if kind == "gqa":
        m = W.Model("stage-gqa", "gqa", 3, 2, 128, 128, 0, "neox", 5e5, 16)
    else:
        m = W.Model("stage-mla", "mla", 2, 1, 576, 64, 512, "interleaved", 1e4, 16)
    wl = W.Workload(f"stage-{kind}", m, lens, reqs, 4, 0)
    ref = Stitched(wl, pool_device="cpu").run()
    try:
        hk = ref.k_pool.cpu().pin_memory()
        hv = ref.v_pool.cpu().pin_memory() if ref.v_pool is not None else None
        dk = torch.zeros_like(ref.k_pool)
        dv = torch.zeros_like(ref.v_pool) if ref.v_pool is not None else None
        distinct, read = pic.pic_pool_read_rows(ref.ctx, ref.plans)
        assert (distinct, read) == (40 + 100 + 20 + 64, 100 + 40 + 20 + 100 + 64 + 50 + 40)
        # in two calls, as a pipelined caller stages request groups: the
        # second skips the rows the first staged
        n = pic.pic_stage_pool(ref.ctx, ref.plans[:1], hk, hv, dk, dv)
        n += pic.pic_stage_pool(ref.ctx, ref.plans[1:], hk, hv, dk, dv, staged_plans=ref.plans[:1])
        row = hk[0, 0].numel() * 2
        assert n == distinct * m.num_layers * row * (2 if hv is not None else 1)
        torch.cuda.synchronize()
        offs = np.concatenate([[0], np.cumsum(lens)[:-1]])
        read_rows = np.zeros(sum(lens), dtype=bool)
        for c, take in {(c, t) for req in reqs for c, t in req}:
            read_rows[offs[c]:offs[c] + take] = True
        for host, staged in ((hk, dk), (hv, dv)):
            if host is None:
                continue
            hb, sb = bits(host), bits(staged)
            assert np.array_equal(sb[:, read_rows], hb[:, read_rows])
            assert not sb[:, ~read_rows].any()
        k_cache = torch.empty_like(ref.k_cache)
        k_cache.view(torch.int16).fill_(-1)
        v_cache = None
        if ref.v_cache is not None:
            v_cache = torch.empty_like(ref.v_cache)
            v_cache.view(torch.int16).fill_(-1)
        ridx, indptr = torch.empty_like(ref.ridx), torch.empty_like(ref.indptr)
        pic.pic_stitch(ref.ctx, ref.plans, dk, dv, k_cache, v_cache, ref.d_bt, ridx, indptr, torch.empty_like(ref.ws))
        torch.cuda.synchronize()
        assert np.array_equal(bits(k_cache), bits(ref.k_cache))
        if v_cache is not None:
            assert np.array_equal(bits(v_cache), bits(ref.v_cache))
        assert torch.equal(ridx, ref.ridx) and torch.equal(indptr, ref.indptr)
        segs, tables, _ = oracle_side(wl, ref.nb)
        want_k, _ = oracle.stitch_paged(bits(hk), None, segs, tables, ref.nb, ref.bs, theta_of(m), pairing_of(m),
                                        m.rope_offset, m.rope_dim)
        assert_k_close(f64(k_cache), want_k, "K from the staged pool")
    finally:
        ref.close()


@pytest.mark.parametrize("kind,n_groups", [("gqa", 1), ("gqa", 2), ("gqa", 3), ("gqa", 9), ("mla", 2), ("mla", 5)])
def test_staged_stitch_equals_the_stitch_from_device_pools(kind, n_groups):
    """pic_stitch_staged (pinned host pools, groups of requests staged on the
    context's copy stream while earlier groups stitch) against pic_stitch
    over the whole pool in device memory: cache rows, recompute list and CSR
    offsets equal bit for bit, one status word clean; the device pool holds
    the rows read and zeros elsewhere.  Five requests reuse chunks across
    groups; 9 groups are clamped to the 5 requests."""
    lens = [40, 17, 100, 33, 9, 64, 5]
    reqs = [[(2, 100), (0, 40)], [(3, 20), (2, 100)], [(5, 64), (2, 50), (0, 40)], [(6, 5), (0, 40)],
            [(3, 33), (5, 64), (6, 5)]]
    if kind == "gqa":
        m = W.Model("staged-gqa", "gqa", 3, 2, 128, 128, 0, "neox", 5e5, 16)
    else:
        m = W.Model("staged-mla", "mla", 2, 1, 576, 64, 512, "interleaved", 1e4, 16)
    wl = W.Workload(f"staged-{kind}", m, lens, reqs, 4, 0)
    ref = Stitched(wl, pool_device="cpu").run()
    try:
        hk = ref.k_pool.cpu().pin_memory()
        hv = ref.v_pool.cpu().pin_memory() if ref.v_pool is not None else None
        dk = torch.zeros_like(ref.k_pool)
        dv = torch.zeros_like(ref.v_pool) if ref.v_pool is not None else None
        k_cache = torch.empty_like(ref.k_cache)
        k_cache.view(torch.int16).fill_(-1)
        v_cache = None
        if ref.v_cache is not None:
            v_cache = torch.empty_like(ref.v_cache)
            v_cache.view(torch.int16).fill_(-1)
        ridx, indptr = torch.full_like(ref.ridx, -7), torch.full_like(ref.indptr, -7)
        ws = torch.empty(pic.pic_stitch_staged_workspace_bytes(ref.ctx, ref.plans, n_groups), dtype=torch.uint8,
                         device=DEV)
        n = pic.pic_stitch_staged(ref.ctx, ref.plans, hk, hv, dk, dv, k_cache, v_cache, ref.d_bt, ridx, indptr, ws,
                                  n_groups=n_groups)
        assert pic.pic_query_device_status(ref.ctx, ws) == 0
        torch.cuda.synchronize()
        distinct, _ = pic.pic_pool_read_rows(ref.ctx, ref.plans)
        row = hk[0, 0].numel() * 2
        assert n == distinct * m.num_layers * row * (2 if hv is not None else 1)
        assert np.array_equal(bits(k_cache), bits(ref.k_cache))
        if v_cache is not None:
            assert np.array_equal(bits(v_cache), bits(ref.v_cache))
        assert torch.equal(ridx, ref.ridx) and torch.equal(indptr, ref.indptr)
        offs = np.concatenate([[0], np.cumsum(lens)[:-1]])
        read_rows = np.zeros(sum(lens), dtype=bool)
        for c, take in {(c, t) for req in reqs for c, t in req}:
            read_rows[offs[c]:offs[c] + take] = True
        assert not read_rows.all()
        for host, staged in ((hk, dk), (hv, dv)):
            if host is not None:
                assert np.array_equal(bits(staged)[:, read_rows], bits(host)[:, read_rows])
                assert not bits(staged)[:, ~read_rows].any()
    finally:
        ref.close()


@pytest.mark.parametrize("seed", range(8))
def test_staged_stitch_on_random_batches(seed):
    """The seeded random batches of the stitch tests (GQA or MLA, either
    pairing, block sizes 1-33, truncated and repeated chunks, recompute
    widths 0-6) through pic_stitch_staged with 1-4 request groups: equal to
    pic_stitch over the device pool, bit for bit."""
    from test_gpu_stitch import _random_workload
    wl = _random_workload(seed)
    ref = Stitched(wl, pool_device="cpu", spare_blocks=2).run()
    try:
        hk = ref.k_pool.cpu().pin_memory()
        hv = ref.v_pool.cpu().pin_memory() if ref.v_pool is not None else None
        dk = torch.zeros_like(ref.k_pool)
        dv = torch.zeros_like(ref.v_pool) if ref.v_pool is not None else None
        k_cache = torch.empty_like(ref.k_cache)
        k_cache.view(torch.int16).fill_(-1)
        v_cache = None
        if ref.v_cache is not None:
            v_cache = torch.empty_like(ref.v_cache)
            v_cache.view(torch.int16).fill_(-1)
        ridx, indptr = torch.full_like(ref.ridx, -7), torch.full_like(ref.indptr, -7)
        n_groups = 1 + seed % 4
        ws = torch.empty(pic.pic_stitch_staged_workspace_bytes(ref.ctx, ref.plans, n_groups), dtype=torch.uint8,
                         device=DEV)
        pic.pic_stitch_staged(ref.ctx, ref.plans, hk, hv, dk, dv, k_cache, v_cache, ref.d_bt, ridx, indptr, ws,
                              n_groups=n_groups)
        assert pic.pic_query_device_status(ref.ctx, ws) == 0
        torch.cuda.synchronize()
        assert np.array_equal(bits(k_cache), bits(ref.k_cache))
        if v_cache is not None:
            assert np.array_equal(bits(v_cache), bits(ref.v_cache))
        assert torch.equal(ridx[:ref.n_rec], ref.ridx[:ref.n_rec]) and torch.equal(indptr, ref.indptr)
    finally:
        ref.close()


def _mixed_context(m, nb):
    """Pool chunks 0-2, chunk B resident in cache blocks 40-42 (40 tokens
    cached at position 300) and chunk C in blocks 44-45 (20 tokens at 50);
    three requests: B mapped at a block boundary, C copied after an odd
    offset, and pool chunks only."""
    ctx = pic.create_from_spec(pic.model_spec_from(m), nb)
    lens, offs = [40, 17, 100], [0, 40, 57]
    ids = [pic.pic_register_chunk(ctx, W.chunk_key("mixed", c), offs[c], lens[c])[0] for c in range(3)]
    b = pic.pic_register_chunk_blocks(ctx, W.chunk_key("mixed", 9), [40, 41, 42], 40, 300)[0]
    c_ = pic.pic_register_chunk_blocks(ctx, W.chunk_key("mixed", 10), [44, 45], 20, 50)[0]
    plans, tables = [], []
    for chunks, alias in (([b, ids[0], ids[2]], True), ([ids[1], c_, ids[0]], False), ([ids[2], ids[1]], False)):
        plan, bt = pic.pic_build_block_table(ctx, chunks, 12, alias=alias, k_nonleading=4)
        plans.append(plan)
        tables.append(bt)
    return ctx, plans, np.stack(tables), sum(lens)


def test_staged_stitch_with_block_resident_and_mapped_chunks():
    """A block-resident chunk mapped into one request (its keys rotated in
    place in the cache, nothing staged) and another copied into a second
    request, beside pool chunks: pic_stitch_staged from a pinned host pool leaves the cache, the
    recompute list and the CSR offsets bit for bit as pic_stitch from the
    device pool does, on two contexts built the same way."""
    m = W.Model("mixed", "gqa", 2, 2, 128, 128, 0, "neox", 1e4, 16)
    nb = 64
    g = torch.Generator().manual_seed(21)
    ctx_a, plans_a, tables, P = _mixed_context(m, nb)
    ctx_b, plans_b, tables_b, _ = _mixed_context(m, nb)
    try:
        assert np.array_equal(tables, tables_b)
        assert pic.pic_plan_segment_mode(plans_a[0], 0) == pic.PIC_SEG_MAPPED
        assert pic.pic_plan_segment_mode(plans_a[1], 1) == pic.PIC_SEG_COPY_BLOCKS
        k_pool = torch.randn((2, P, 2, 128), generator=g).to(torch.bfloat16)
        v_pool = torch.randn((2, P, 2, 128), generator=g).to(torch.bfloat16)
        cache_k = torch.randn((2, nb, 16, 2, 128), generator=g).to(torch.bfloat16)
        cache_v = torch.randn((2, nb, 16, 2, 128), generator=g).to(torch.bfloat16)
        bt = torch.from_numpy(tables).to(DEV)
        n_rec = sum(pic.pic_plan_info(p)["num_recompute"] for p in plans_a)
        outs = []
        for ctx, plans, staged in ((ctx_a, plans_a, False), (ctx_b, plans_b, True)):
            kc, vc = cache_k.to(DEV), cache_v.to(DEV)
            ridx = torch.full((n_rec,), -7, dtype=torch.int32, device=DEV)
            indptr = torch.full((4,), -7, dtype=torch.int32, device=DEV)
            if staged:
                dk, dv = torch.zeros((2, P, 2, 128), dtype=torch.bfloat16, device=DEV), torch.zeros(
                    (2, P, 2, 128), dtype=torch.bfloat16, device=DEV)
                ws = torch.empty(pic.pic_stitch_staged_workspace_bytes(ctx, plans, 2), dtype=torch.uint8, device=DEV)
                pic.pic_stitch_staged(ctx, plans, k_pool.pin_memory(), v_pool.pin_memory(), dk, dv, kc, vc, bt, ridx,
                                      indptr, ws, n_groups=2)
            else:
                ws = torch.empty(pic.pic_workspace_bytes(ctx, plans), dtype=torch.uint8, device=DEV)
                pic.pic_stitch(ctx, plans, k_pool.to(DEV), v_pool.to(DEV), kc, vc, bt, ridx, indptr, ws)
            assert pic.pic_query_device_status(ctx, ws) == 0
            torch.cuda.synchronize()
            outs.append((bits(kc), bits(vc), ridx.cpu(), indptr.cpu()))
        (ka, va, ra, ia), (kb, vb, rb, ib) = outs
        assert np.array_equal(ka, kb) and np.array_equal(va, vb)
        assert torch.equal(ra, rb) and torch.equal(ia, ib)
        # the mapped chunk's keys moved in place: blocks 40-42 changed
        assert not np.array_equal(ka[:, 40:43], bits(cache_k)[:, 40:43])
    finally:
        pic.pic_destroy(ctx_a)
        pic.pic_destroy(ctx_b)


def test_serving_stress_full_size_staged():
    """The benchmark's end-to-end launch at full size: the serving-stress pool
    (61 GB of K and V) in pinned host memory, staged by pic_stitch_staged in
    32 request groups into a cleared device pool and stitched into the
    137 GB cache.  Sampled rows against the oracle (keys per element within
    the contract, values bit for bit), the staged rows equal to the host rows,
    the recompute list exact, and the staged bytes the distinct rows read."""
    from test_gpu_stitch import _check_sampled, _sample_rows
    wl = W.serving_stress()
    st = Stitched(wl)
    try:
        hk = torch.empty(st.k_pool.shape, dtype=st.k_pool.dtype, pin_memory=True)
        hk.copy_(st.k_pool)
        hv = torch.empty(st.v_pool.shape, dtype=st.v_pool.dtype, pin_memory=True)
        hv.copy_(st.v_pool)
        st.k_pool.zero_()
        st.v_pool.zero_()
        ws = torch.empty(pic.pic_stitch_staged_workspace_bytes(st.ctx, st.plans, 32), dtype=torch.uint8, device=DEV)
        n = pic.pic_stitch_staged(st.ctx, st.plans, hk, hv, st.k_pool, st.v_pool, st.k_cache, st.v_cache, st.d_bt,
                                  st.ridx, st.indptr, ws, n_groups=32)
        assert pic.pic_query_device_status(st.ctx, ws) == 0
        torch.cuda.synchronize()
        distinct, read = pic.pic_pool_read_rows(st.ctx, st.plans)
        assert read == wl.token_layers // wl.model.num_layers and distinct < read
        assert n == distinct * wl.model.num_layers * 2048 * 2
        segs, tables, rec = oracle_side(wl, st.nb)
        _check_sampled(st, segs, tables, 6000, 5)
        l_idx, _, _, src, _ = _sample_rows(st, segs, tables, 6000, 5)
        li, si = l_idx.cpu(), src.cpu()
        assert np.array_equal(bits(st.k_pool[l_idx, src]), bits(hk[li, si]))
        assert np.array_equal(bits(st.v_pool[l_idx, src]), bits(hv[li, si]))
        indptr, idx = oracle.recompute_csr(rec)
        assert st.indptr.cpu().tolist() == indptr.tolist()
        assert st.ridx.cpu().numpy()[:st.n_rec].tolist() == idx.tolist()
    finally:
        st.close()
        del st
        torch.cuda.empty_cache()


def test_stage_pool_over_more_ranges_than_one_launch_takes():
    """1,100 chunks of 2 tokens, one request taking the first token of each:
    1,100 separate row ranges, so the copy runs as two launches (1,024 ranges
    each at most).  Every first row arrives, every second row stays zero."""
    n = 1100
    m = W.Model("stage-many", "gqa", 2, 1, 64, 64, 0, "neox", 1e4, 16)
    wl = W.Workload("stage-many", m, [2] * n, [[(c, 1) for c in range(n)]], 0, 0)
    ref = Stitched(wl, pool_device="cpu")
    try:
        assert pic.pic_pool_read_rows(ref.ctx, ref.plans) == (n, n)
        hk = ref.k_pool.cpu().pin_memory()
        hv = ref.v_pool.cpu().pin_memory()
        dk, dv = torch.zeros_like(ref.k_pool), torch.zeros_like(ref.v_pool)
        got = pic.pic_stage_pool(ref.ctx, ref.plans, hk, hv, dk, dv)
        assert got == n * 2 * 128 * 2   # rows x layers x row bytes x (K, V)
        torch.cuda.synchronize()
        for host, staged in ((hk, dk), (hv, dv)):
            hb, sb = bits(host), bits(staged)
            assert np.array_equal(sb[:, 0::2], hb[:, 0::2])
            assert not sb[:, 1::2].any()
    finally:
        ref.close()


def test_stage_pool_refuses_pageable_and_swapped_pointers():
    lens = [40, 17]
    m = W.Model("stage-bad", "gqa", 2, 2, 128, 128, 0, "neox", 1e4, 16)
    wl = W.Workload("stage-bad", m, lens, [[(0, 40), (1, 17)]], 4, 0)
    ref = Stitched(wl, pool_device="cpu")
    try:
        hk = ref.k_pool.cpu().pin_memory()
        hv = ref.v_pool.cpu().pin_memory()
        L = pic.load()
        arr = pic._plan_array(ref.plans)
        ls = hk.stride(0) * 2
        pageable = ref.k_pool.cpu()
        for args in ((pageable, hv, ref.k_pool, ref.v_pool),     # pageable host pool
                     (ref.k_pool, ref.v_pool, ref.k_pool, ref.v_pool),  # device memory as the host pool
                     (hk, hv, hk, hv)):                          # host memory as the device pool
            st = L.pic_stage_pool(ref.ctx, arr, len(ref.plans), None, 0, ctypes.c_void_p(args[0].data_ptr()),
                                  ctypes.c_void_p(args[1].data_ptr()), ls, ctypes.c_void_p(args[2].data_ptr()),
                                  ctypes.c_void_p(args[3].data_ptr()), ls, None, None)
            assert pic.STATUS_NAMES[st] == "PIC_ERR_INVALID_ARG", args
    finally:
        ref.close()


def test_host_cache_in_place_shift():
    m = W.Model("ip-host", "gqa", 2, 2, 128, 128, 0, "neox", 1e4, 16)
    ctx = pic.create_from_spec(pic.model_spec_from(m), 8)
    try:
        cache = torch.empty((2, 8, 16, 2, 128), dtype=torch.bfloat16)
        W.fill_random_bf16(cache, 9, "host-inplace")
        host = cache.pin_memory()
        devc = cache.to(DEV)
        tables = [[3, 1, 6, 0]]
        bt = torch.tensor(tables, dtype=torch.int32, device=DEV)
        segs = [(0, 2, 30, 4097), (0, 40, 9, -3)]
        ws = torch.empty(pic.pic_rerotate_workspace_bytes(ctx, segs), dtype=torch.uint8, device=DEV)
        pic.pic_rerotate_inplace(ctx, host, bt, segs, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0
        pic.pic_rerotate_inplace(ctx, devc, bt, segs, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0
        assert np.array_equal(bits(host), bits(devc))
        want = oracle.rerotate_inplace(bits(cache), tables, segs, 16, oracle.rope_inv_freq(128, 1e4),
                                       oracle.NEOX_HALF, 0, 128)
        assert_k_close(f64(host), want, "host in place")
    finally:
        pic.pic_destroy(ctx)


def test_pageable_host_memory_is_refused_before_launch():
    m = W.Model("pageable", "gqa", 1, 1, 64, 64, 0, "neox", 1e4, 16)
    ctx = pic.create_from_spec(pic.model_spec_from(m), 2)
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("p", 0), 0, 10)
        plan, bt = pic.pic_build_block_table(ctx, [0], 1)
        pageable = np.zeros((1, 16, 1, 64), dtype=np.uint16)   # plain numpy memory, not pinned
        dcache = torch.empty((1, 2, 16, 1, 64), dtype=torch.bfloat16, device=DEV)
        d_bt = torch.from_numpy(bt).to(DEV).view(1, -1)
        ws = torch.empty(pic.pic_workspace_bytes(ctx, [plan]), dtype=torch.uint8, device=DEV)
        arr = pic._plan_array([plan])
        p = ctypes.c_void_p(pageable.ctypes.data)
        L = pic.load()
        st = L.pic_stitch(ctx, arr, 1, p, p, 16 * 64 * 2, ctypes.c_void_p(dcache.data_ptr()),
                          ctypes.c_void_p(dcache.data_ptr()), dcache.stride(0) * 2, ctypes.c_void_p(d_bt.data_ptr()),
                          1, None, None, 0, ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
        assert pic.STATUS_NAMES[st] == "PIC_ERR_INVALID_ARG"
        assert "pageable" in pic.pic_last_error(ctx)
    finally:
        pic.pic_destroy(ctx)
