"""pic_stitch_noalloc against pic_stitch, through the C ABI.

pic_stitch_noalloc serves callers that may not allocate device memory where
they stitch (an engine whose KV-cache pool already owns the HBM, a plugin
that only receives its input and output tensors, a loop that must not pay
for cudaMalloc/cudaFree).  It runs the same kernel with the library's own fixed
device scratch instead of a caller workspace, so its output must equal
pic_stitch's on the same inputs bit for bit -- checked here on two calls in
a row with different batches, so the second call also shows that leftovers
from the first call in the shared scratch do not leak into its result.  The
first call is also compared with the oracle, and a call that raises the
device status word is followed by a clean one that must report 0.

This file is named to be collected last: a failure here leaves every other
test already run.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import assert_k_close, bits, oracle_side, pairing_of, sentinel_like, theta_of
from position_independent_kv_stitch_gb300 import pic

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(wl, bs_blocks_extra=0):
    m = wl.model
    bs = m.block_size
    nb = sum(-(-t // bs) for t in wl.request_tokens) + bs_blocks_extra
    mb = max(-(-t // bs) for t in wl.request_tokens)
    ctx = pic.create_from_spec(pic.model_spec_from(m), nb)
    ids = [pic.pic_register_chunk(ctx, W.chunk_key(wl.name, c), off, n)[0]
           for c, (off, n) in enumerate(zip(wl.pool_offsets, wl.chunk_lens))]
    plans, tables = [], []
    for req in wl.requests:
        plan, bt = pic.pic_build_block_table(ctx, [ids[c] for c, _ in req], mb, take_tokens=[t for _, t in req],
                                             k_nonleading=wl.k_nonleading, k_leading=wl.k_leading)
        plans.append(plan)
        tables.append(bt)
    k_pool = W.make_pool(wl, "k", device="cpu").to(DEV)
    v_pool = W.make_pool(wl, "v", device="cpu").to(DEV) if m.kind == "gqa" else None
    return ctx, m, nb, plans, torch.from_numpy(np.stack(tables)).to(DEV), k_pool, v_pool


def _outputs(m, nb, n_req, n_rec):
    shape = (m.num_layers, nb, m.block_size) + tuple(m.row_shape)
    k = sentinel_like(shape, DEV)
    v = sentinel_like(shape, DEV) if m.kind == "gqa" else None
    ridx = torch.full((max(1, n_rec),), -7, dtype=torch.int32, device=DEV)
    indptr = torch.full((n_req + 1,), -7, dtype=torch.int32, device=DEV)
    return k, v, ridx, indptr


def _compare(wl, against_oracle=False):
    """pic_stitch_noalloc against pic_stitch on the same inputs: the same
    kernel runs on the same inputs, so every output must be bit-identical.
    Optionally also against the oracle, at the contract tolerance."""
    ctx, m, nb, plans, d_bt, k_pool, v_pool = _setup(wl)
    try:
        n_rec = len(pic.pic_recompute_indices(plans)[1])
        ka, va, ia, pa = _outputs(m, nb, len(plans), n_rec)
        ws = torch.empty(pic.pic_workspace_bytes(ctx, plans), dtype=torch.uint8, device=DEV)
        pic.pic_stitch(ctx, plans, k_pool, v_pool, ka, va, d_bt, ia, pa, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0

        kb, vb, ib, pb = _outputs(m, nb, len(plans), n_rec)
        status = torch.full((1,), 77, dtype=torch.int32, device=DEV)
        pic.pic_stitch_noalloc(ctx, plans, k_pool, v_pool, kb, vb, d_bt, ib, pb, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0

        assert np.array_equal(bits(ka), bits(kb))
        if va is not None:
            assert np.array_equal(bits(va), bits(vb))
        assert torch.equal(ia, ib) and torch.equal(pa, pb)

        if against_oracle:
            segs, tables, rec = oracle_side(wl, nb)
            assert d_bt.cpu().numpy()[:, :len(tables[0])].tolist()[0] == tables[0]
            want_k, want_v = oracle.stitch_paged(bits(k_pool), None if v_pool is None else bits(v_pool), segs,
                                                 tables, nb, m.block_size, theta_of(m), pairing_of(m),
                                                 m.rope_offset, m.rope_dim)
            assert_k_close(kb.float().cpu().double().numpy(), want_k, "K (no-alloc)")
            if want_v is not None:
                assert np.array_equal(bits(vb), want_v)
            flat = [p for r in rec for p in r]
            assert ib.cpu().numpy()[:len(flat)].tolist() == flat
    finally:
        pic.pic_destroy(ctx)


def test_noalloc_matches_pic_stitch_two_calls_in_a_row():
    # call 1: the tiny GQA request, also checked against the oracle;
    # call 2: a two-request ragged MLA batch
    _compare(W.tiny_gqa(), against_oracle=True)
    base = W.deepseek_v3_mla(context_tokens=700, num_layers=2)
    reqs = [base.requests[0], list(reversed(base.requests[0][5:40]))]
    _compare(W.Workload("noalloc-mla", base.model, base.chunk_lens, reqs, 4, 32))


def test_noalloc_status_word_starts_clean_on_every_call():
    """The shared scratch keeps the last call's contents, status word
    included.  Call 1 has a block-table entry outside the cache, which the
    kernel's own bounds check skips and reports; call 2, clean, must report
    0 and match pic_stitch bit for bit."""
    wl = W.tiny_gqa()
    ctx, m, nb, plans, d_bt, k_pool, v_pool = _setup(wl)
    try:
        n_rec = len(pic.pic_recompute_indices(plans)[1])
        bad_bt = d_bt.clone()
        bad_bt[0, 3] = nb            # one entry outside [0, nb)
        k1, v1, i1, p1 = _outputs(m, nb, 1, n_rec)
        status = torch.zeros((1,), dtype=torch.int32, device=DEV)
        pic.pic_stitch_noalloc(ctx, plans, k_pool, v_pool, k1, v1, bad_bt, i1, p1, status=status)
        torch.cuda.synchronize()
        assert status.item() & pic.PIC_DEV_BAD_BLOCK

        # the same plans again (stitching copies never consume a plan), clean table
        k2, v2, i2, p2 = _outputs(m, nb, 1, n_rec)
        status.fill_(77)
        pic.pic_stitch_noalloc(ctx, plans, k_pool, v_pool, k2, v2, d_bt, i2, p2, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0

        ka, va, ia, pa = _outputs(m, nb, 1, n_rec)
        ws = torch.empty(pic.pic_workspace_bytes(ctx, plans), dtype=torch.uint8, device=DEV)
        pic.pic_stitch(ctx, plans, k_pool, v_pool, ka, va, d_bt, ia, pa, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0
        assert np.array_equal(bits(ka), bits(k2)) and np.array_equal(bits(va), bits(v2))
        assert torch.equal(ia, i2) and torch.equal(pa, p2)
    finally:
        pic.pic_destroy(ctx)


def test_noalloc_rejects_batch_beyond_scratch():
    m = W.Model("big", "gqa", 1, 1, 64, 64, 0, "neox", 1e4, 1)
    ctx = pic.create_from_spec(pic.model_spec_from(m), 200000)
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("big", 0), 0, 150000)
        plan, bt = pic.pic_build_block_table(ctx, [0], 150000)   # 150,000 one-token runs > 4 MiB
        d_bt = torch.from_numpy(bt).to(DEV).view(1, -1)
        pool = torch.zeros((1, 16, 1, 64), dtype=torch.bfloat16, device=DEV)
        with pytest.raises(pic.PicError) as e:
            pic.pic_stitch_noalloc(ctx, [plan], pool, pool, pool, pool, d_bt)
        assert e.value.status_name == "PIC_ERR_CAPACITY"
        assert "static scratch" in str(e.value)
    finally:
        pic.pic_destroy(ctx)
