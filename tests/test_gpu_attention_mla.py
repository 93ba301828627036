"""GPU parity of decode attention for MLA models (Irminsul 2.1-2.2): every
query head reads the same latent rows, row = [cKV (512) | k_r (64)]; a chunk's
k_r is rotated by its delta on the way in, the latent is used as stored and is
the value.  Against the fp64 oracle's attention over exactly rotated rows."""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import bits, random_attend_layout, register_attend_layout
from position_independent_kv_stitch_gb300 import pic

pytestmark = pytest.mark.gpu
DEV = "cuda"
LATENT, ROPE = 512, 64
ROW = LATENT + ROPE

_POOL_LENS = [1, 5, 16, 17, 33, 100, 250, 300, 64, 128, 7, 400]
_BLOCK_CHUNK = (45, [190, 191, 192], 700)   # tokens, blocks, position its keys sit at


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pic.load(build_if_missing=True)


@pytest.fixture(params=["tc", "mma"], autouse=True)
def attend_kernel(request, monkeypatch):
    """Every case runs on both MLA attention kernels, chosen at pic_create:
    tcgen05 with TMEM accumulators (the default) and warp-level mma.sync."""
    monkeypatch.setenv("PIC_ATTEND_KERNEL", request.param)
    return request.param


def _check_variant(ctx, kernel):
    want = pic.PIC_VARIANT_TENSOR_CORE_TMEM if kernel == "tc" else pic.PIC_VARIANT_WARP_MMA
    assert pic.pic_kernel_variant(ctx, 2) == want


def _setup(pairing, L, seed, rep=1, row_scale=None):
    bs, nb = 16, 200 + 120 * (rep - 1)
    m = W.Model("attn-mla", "mla", L, 1, ROW, ROPE, LATENT, pairing, 1e4, bs)
    ctx = pic.create_from_spec(pic.model_spec_from(m), nb)
    _check_variant(ctx, os.environ["PIC_ATTEND_KERNEL"])
    offs = [0]
    for n in _POOL_LENS[:-1]:
        offs.append(offs[-1] + n)
    ids, sources = [], {}
    for c, (o, n) in enumerate(zip(offs, _POOL_LENS)):
        cid = pic.pic_register_chunk(ctx, W.chunk_key("attn-mla", c), o, n)[0]
        ids.append(cid)
        sources[cid] = ("pool", o)
    n_b, blocks, base = _BLOCK_CHUNK
    bid = pic.pic_register_chunk_blocks(ctx, W.chunk_key("attn-mla", 99), blocks, n_b, base)[0]
    sources[bid] = ("blocks", blocks)
    g = torch.Generator().manual_seed(seed)
    P = offs[-1] + _POOL_LENS[-1]
    pool = torch.randn((L, P, ROW), generator=g)
    for c, f in (row_scale or {}).items():  # chunk index -> factor on its pool rows
        pool[:, offs[c]:offs[c] + _POOL_LENS[c]] *= f
    pool = pool.to(torch.bfloat16)
    cache = torch.randn((L, nb, bs, ROW), generator=g).to(torch.bfloat16)

    def positions(chunks, start, gaps):
        pos, p = [], start
        for j, c in enumerate(chunks):
            p += gaps.get(j, 0)
            pos.append(p)
            p += n_b if c == bid else _POOL_LENS[ids.index(c)]
        return pos, p

    pool_runs = [ids[9], ids[3], ids[8], ids[0], ids[4], ids[10], ids[6], ids[1]]
    specs = [([ids[5], ids[11], ids[2], bid, ids[7]] + [ids[7], ids[4]] * (rep - 1), 3, {4: 10}, 6),
             (pool_runs * rep, 0, {}, 0),
             ([ids[11], ids[6], ids[5]] * rep, 0, {}, 40)]
    plans, tables = [], []
    for chunks, start, gaps, tail in specs:
        pos, end = positions(chunks, start, gaps)
        plan, bt = pic.pic_build_block_table(ctx, chunks, 64 * rep, dst_pos=pos, start_pos=start,
                                             total_tokens=end + tail, k_nonleading=4)
        plans.append(plan)
        tables.append(bt)
    return dict(m=m, ctx=ctx, plans=plans, tables=tables, sources=sources, pool=pool, cache=cache, bs=bs, L=L)


def _context_rows(S, r):
    """fp64 latent rows of request r's context, rope slice exactly rotated."""
    m, bs = S["m"], S["bs"]
    theta = oracle.model_inv_freq(ROPE, m.rope_theta, None)
    pairing = oracle.NEOX_HALF if m.pairing == "neox" else oracle.INTERLEAVED
    plan, table = S["plans"][r], S["tables"][r]
    T = pic.pic_plan_info(plan)["total_tokens"]
    pos = np.arange(T)
    blk_i = torch.as_tensor(np.asarray(table)[pos // bs], dtype=torch.long)
    row_i = torch.as_tensor(pos % bs, dtype=torch.long)
    rows = oracle.bf16_bits_to_f64(bits(S["cache"][:, blk_i, row_i]))
    segs = []
    for j in range(pic.pic_plan_info(plan)["num_segments"]):
        sg = pic.pic_plan_segment(plan, j)
        n, p0 = sg["num_tokens"], sg["dst_pos"]
        kind, where = S["sources"][sg["chunk_id"]]
        t = np.arange(n)
        if kind == "pool":
            src = S["pool"][:, torch.as_tensor(sg["src_tok"] + t, dtype=torch.long)]
        else:
            blk = torch.as_tensor(np.asarray(where)[t // bs], dtype=torch.long)
            src = S["cache"][:, blk, torch.as_tensor(t % bs, dtype=torch.long)]
        rows[:, p0:p0 + n] = oracle.rotate_rows(oracle.bf16_bits_to_f64(bits(src)), sg["delta"], theta, pairing,
                                                LATENT, ROPE)
        segs.append(oracle.Segment(sg["chunk_id"], sg["src_tok"], n, p0, sg["delta"]))
    return rows, segs, T


def _check_over_cache(S, cache, q, out, lse, scale, bias_value, atol):
    """Against the oracle over the rows as the cache holds them after a
    stitch (bf16, rope slices already rotated): what the cache path reads."""
    qb, bs = bits(q), S["bs"]
    cb = oracle.bf16_bits_to_f64(bits(cache))
    for r in range(3):
        _, segs, T = _context_rows(S, r)
        table = np.asarray(S["tables"][r])
        pos = np.arange(T)
        rows = cb[:, table[pos // bs], pos % bs]
        bias = oracle.sink_bias(segs, T, 4, bias_value) if bias_value else None
        for l in range(S["L"]):
            o, sv = oracle.attention_decode(oracle.bf16_bits_to_f64(qb[l, r]), rows[l][:, None, :],
                                            rows[l][:, None, :LATENT], scale, bias)
            np.testing.assert_allclose(out[l, r], o, atol=atol, rtol=0)
            np.testing.assert_allclose(lse[l, r], sv, atol=atol, rtol=0)


def _attend(S, H, source, bias_value, pool=None, cache=None):
    L = S["L"]
    g = torch.Generator().manual_seed(5)
    q = torch.randn((L, 3, H, ROW), generator=g).to(torch.bfloat16)
    out = torch.empty((L, 3, H, LATENT), dtype=torch.float32, device=DEV)
    lse = torch.empty((L, 3, H), dtype=torch.float32, device=DEV)
    ws = torch.empty(pic.pic_attend_workspace_bytes(S["ctx"], S["plans"], H, L), dtype=torch.uint8, device=DEV)
    scale = 1.0 / math.sqrt(192)
    pool = S["pool"].to(DEV) if pool is None else pool
    cache = S["cache"].to(DEV) if cache is None else cache
    pic.pic_attend_decode(S["ctx"], S["plans"], source, q.to(DEV), scale, pool, None, cache, None, out, lse, ws,
                          sink_bias=bias_value)
    assert pic.pic_query_device_status(S["ctx"], ws) == 0
    return q, out.cpu().double().numpy(), lse.cpu().double().numpy(), scale


def _check_against_oracle(S, q, out, lse, scale, bias_value, atol):
    qb = bits(q)
    for r in range(3):
        rows, segs, T = _context_rows(S, r)
        bias = oracle.sink_bias(segs, T, 4, bias_value) if bias_value else None
        for l in range(S["L"]):
            keys = rows[l][:, None, :]
            vals = rows[l][:, None, :LATENT]
            o, s = oracle.attention_decode(oracle.bf16_bits_to_f64(qb[l, r]), keys, vals, scale, bias)
            np.testing.assert_allclose(out[l, r], o, atol=atol, rtol=0)
            np.testing.assert_allclose(lse[l, r], s, atol=atol, rtol=0)


@pytest.mark.parametrize("pairing,H,L,bias_value,rep", [
    ("interleaved", 16, 2, -15.0, 1),
    ("interleaved", 16, 2, 0.0, 4),
    ("neox", 16, 2, -15.0, 1),
    ("interleaved", 32, 2, 0.0, 1),
    ("neox", 32, 2, -15.0, 3),
    ("interleaved", 64, 1, -15.0, 1),
    ("interleaved", 128, 1, 0.0, 1),
])
def test_fused_mla_attention_matches_oracle(pairing, H, L, bias_value, rep):
    """Three requests of 250-1,400 positions (times rep): chunks of 1..400
    tokens, inline gaps and a trailing run of inline tokens, a block-resident
    chunk read from its blocks, delta 0 and nonzero; every (layer, request,
    query head) against the oracle.  64 and 128 heads run as 2 and 4 head
    groups of 32 per request."""
    S = _setup(pairing, L, seed=4, rep=rep)
    try:
        q, out, lse, scale = _attend(S, H, pic.PIC_ATTEND_FUSED, bias_value)
        _check_against_oracle(S, q, out, lse, scale, bias_value, 2e-3)
    finally:
        pic.pic_destroy(S["ctx"])


@pytest.mark.parametrize("H", [16, 32])
def test_mla_running_max_rises_in_a_later_tile(H):
    """Rows of chunks 6 and 11 scaled by 6 and of chunks 9, 3 and 8 by 1/4,
    in contexts 16 times the base case (about 1,700 stages, so each of the
    152 CTAs takes about 11 and several tiles of a key): where a CTA's range
    runs from small rows into scaled ones, a later tile's scores pass the
    running max by far more than the lazy threshold (8 in log2 units), and
    the O and l already accumulated are rescaled (about 150 such tiles in a
    CPU model of the split; random rows of one scale never get there).
    Outputs reach about 6 in magnitude."""
    S = _setup("interleaved", 1, seed=12, rep=16, row_scale={6: 6.0, 11: 6.0, 9: 0.25, 3: 0.25, 8: 0.25})
    try:
        q, out, lse, scale = _attend(S, H, pic.PIC_ATTEND_FUSED, -15.0)
        assert np.abs(out).max() > 2.0  # the scaled rows dominate
        _check_against_oracle(S, q, out, lse, scale, -15.0, 4e-3)
    finally:
        pic.pic_destroy(S["ctx"])


def test_mla_cache_path_over_materialized_stitch():
    """Stitch the requests into the cache (MLA stitch: latent copied, rope
    rotated, rounded to bf16 once), then attend from the cache: the oracle
    over the stitched rows at the attention tolerance, the oracle over
    exactly rotated rows up to that rounding, and the fused path closer."""
    S = _setup("interleaved", 2, seed=6)
    try:
        ctx = S["ctx"]
        cache = S["cache"].to(DEV)
        pool = S["pool"].to(DEV)
        d_bt = torch.from_numpy(np.stack(S["tables"])).to(DEV)
        ws = torch.empty(pic.pic_workspace_bytes(ctx, S["plans"]), dtype=torch.uint8, device=DEV)
        pic.pic_stitch(ctx, S["plans"], pool, None, cache, None, d_bt, None, None, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0
        q, out_c, lse_c, scale = _attend(S, 16, pic.PIC_ATTEND_CACHE, -15.0, pool, cache)
        _, out_f, lse_f, _ = _attend(S, 16, pic.PIC_ATTEND_FUSED, -15.0, pool, cache)
        # the cache path against the oracle over the GPU-stitched rows it reads
        _check_over_cache(S, cache, q, out_c, lse_c, scale, -15.0, 2e-3)
        # both against exactly rotated rows; the cache path's rows were rounded once
        _check_against_oracle(S, q, out_f, lse_f, scale, -15.0, 2e-3)
        _check_against_oracle(S, q, out_c, lse_c, scale, -15.0, 3e-2)
    finally:
        pic.pic_destroy(S["ctx"])


def _random_setup(seed):
    """A seeded random MLA context: either pairing, 1-3 layers, block size
    1-33, rope theta 1e4 or 1e6, and the chunk and request mix of
    random_attend_layout."""
    rng = np.random.default_rng(5000 + seed)
    pairing = ["neox", "interleaved"][int(rng.integers(2))]
    L = int(rng.integers(1, 4))
    bs = int(rng.choice([1, 4, 16, 33]))
    m = W.Model(f"attn-mla-rand-{seed}", "mla", L, 1, ROW, ROPE, LATENT, pairing, float(rng.choice([1e4, 1e6])), bs)
    lay = random_attend_layout(rng, bs)
    ctx = pic.create_from_spec(pic.model_spec_from(m), lay["nb"])
    _check_variant(ctx, os.environ["PIC_ATTEND_KERNEL"])
    plans, tables, sources = register_attend_layout(ctx, lay, m.name, bs)
    g = torch.Generator().manual_seed(seed)
    pool = torch.randn((L, lay["P"], ROW), generator=g).to(torch.bfloat16)
    cache = torch.randn((L, lay["nb"], bs, ROW), generator=g).to(torch.bfloat16)
    return dict(m=m, ctx=ctx, plans=plans, tables=tables, sources=sources, pool=pool, cache=cache, bs=bs, L=L,
                k=lay["k"], rng=rng)


@pytest.mark.parametrize("seed", range(8))
def test_random_mla_contexts_match_oracle(seed):
    """Seeded random contexts (block sizes, chunk lengths, block-resident
    chunks, repeats, truncation, inline gaps, pseudo-sink widths, 16-128
    heads, a random layer window) on both MLA kernels: fused against the
    oracle over exactly rotated rows, the cache path against the oracle over
    the cache rows as stored; every (layer, request, query head) within
    2e-3."""
    S = _random_setup(seed)
    try:
        rng, ctx, plans, bs = S["rng"], S["ctx"], S["plans"], S["bs"]
        L, n = S["L"], len(plans)
        H = int(rng.choice([16, 32, 64, 128]))
        bias_value = -15.0 if rng.random() < 0.5 else 0.0
        lb = int(rng.integers(0, L))
        nl = int(rng.integers(1, L - lb + 1))
        q = torch.randn((nl, n, H, ROW), generator=torch.Generator().manual_seed(60 + seed)).to(torch.bfloat16)
        qb = bits(q)
        scale = 1.0 / math.sqrt(192)
        pool, cache = S["pool"].to(DEV), S["cache"].to(DEV)
        ws = torch.empty(pic.pic_attend_workspace_bytes(ctx, plans, H, nl), dtype=torch.uint8, device=DEV)
        cache_rows = oracle.bf16_bits_to_f64(bits(S["cache"]))
        for source in (pic.PIC_ATTEND_FUSED, pic.PIC_ATTEND_CACHE):
            out = torch.full((nl, n, H, LATENT), float("nan"), dtype=torch.float32, device=DEV)
            lse = torch.full((nl, n, H), float("nan"), dtype=torch.float32, device=DEV)
            pic.pic_attend_decode(ctx, plans, source, q.to(DEV), scale, pool, None, cache, None, out, lse, ws,
                                  sink_bias=bias_value, layer_begin=lb)
            assert pic.pic_query_device_status(ctx, ws) == 0
            out, lse = out.cpu().double().numpy(), lse.cpu().double().numpy()
            for r in range(n):
                rows, segs, T = _context_rows(S, r)
                if source == pic.PIC_ATTEND_CACHE:
                    pos = np.arange(T)
                    rows = cache_rows[:, np.asarray(S["tables"][r])[pos // bs], pos % bs]
                bias = oracle.sink_bias(segs, T, S["k"], bias_value) if bias_value else None
                for i in range(nl):
                    x = rows[lb + i]
                    o, sv = oracle.attention_decode(oracle.bf16_bits_to_f64(qb[i, r]), x[:, None, :],
                                                    x[:, None, :LATENT], scale, bias)
                    np.testing.assert_allclose(out[i, r], o, atol=2e-3, rtol=0, err_msg=f"source {source} r {r} l {i}")
                    np.testing.assert_allclose(lse[i, r], sv, atol=2e-3, rtol=0, err_msg=f"source {source} r {r} l {i}")
    finally:
        pic.pic_destroy(S["ctx"])


def test_mla_attention_over_a_layer_window():
    """Layers [1, 3) of a 3-layer model in one call: q, out and lse hold the
    window's layers only, while the pool and cache rows are read from
    absolute layers 1 and 2 (the tcgen05 kernel's TMA layer coordinate and
    its query indexing differ by layer_begin)."""
    S = _setup("interleaved", 3, seed=8)
    try:
        H, lb, nl = 16, 1, 2
        g = torch.Generator().manual_seed(9)
        q = torch.randn((nl, 3, H, ROW), generator=g).to(torch.bfloat16)
        out = torch.empty((nl, 3, H, LATENT), dtype=torch.float32, device=DEV)
        lse = torch.empty((nl, 3, H), dtype=torch.float32, device=DEV)
        ws = torch.empty(pic.pic_attend_workspace_bytes(S["ctx"], S["plans"], H, nl), dtype=torch.uint8, device=DEV)
        scale = 1.0 / math.sqrt(192)
        pic.pic_attend_decode(S["ctx"], S["plans"], pic.PIC_ATTEND_FUSED, q.to(DEV), scale, S["pool"].to(DEV), None,
                              S["cache"].to(DEV), None, out, lse, ws, sink_bias=-15.0, layer_begin=lb)
        assert pic.pic_query_device_status(S["ctx"], ws) == 0
        out, lse, qb = out.cpu().double().numpy(), lse.cpu().double().numpy(), bits(q)
        for r in range(3):
            rows, segs, T = _context_rows(S, r)
            bias = oracle.sink_bias(segs, T, 4, -15.0)
            for l in range(nl):
                o, sv = oracle.attention_decode(oracle.bf16_bits_to_f64(qb[l, r]), rows[lb + l][:, None, :],
                                                rows[lb + l][:, None, :LATENT], scale, bias)
                np.testing.assert_allclose(out[l, r], o, atol=2e-3, rtol=0)
                np.testing.assert_allclose(lse[l, r], sv, atol=2e-3, rtol=0)
    finally:
        pic.pic_destroy(S["ctx"])


def test_mla_rejects_unsupported_head_counts():
    S = _setup("interleaved", 1, seed=7)
    try:
        with pytest.raises(pic.PicError) as e:
            _attend(S, 24, pic.PIC_ATTEND_FUSED, 0.0)
        assert e.value.status_name == "PIC_ERR_UNSUPPORTED"
    finally:
        pic.pic_destroy(S["ctx"])


@pytest.mark.parametrize("H", [16, 32])
def test_deepseek_full_launch_sampled_layers(H):
    """The benchmark's launch (DeepSeek-V3 MLA shapes: 61 layers, 65,536
    positions of 16-128-token chunks behind a 32-token leading chunk, 16 or
    32 query heads: the query-rotating and the key-rotating kernel) in one
    call; layers 0, 30 and 60 against the oracle, and the cache path over the
    stitched copy against the fused result everywhere."""
    from gpu_util import Stitched
    wl = W.deepseek_v3_mla()
    st = Stitched(wl).run()
    try:
        _check_variant(st.ctx, os.environ["PIC_ATTEND_KERNEL"])
        m = wl.model
        L = m.num_layers
        g = torch.Generator(device=DEV)
        g.manual_seed(11)
        q = torch.empty((L, 1, H, ROW), dtype=torch.bfloat16, device=DEV).normal_(0.0, 1.0, generator=g)
        scale = 1.0 / math.sqrt(192)
        ws = torch.empty(pic.pic_attend_workspace_bytes(st.ctx, st.plans, H, L), dtype=torch.uint8, device=DEV)
        res = {}
        for src in (pic.PIC_ATTEND_FUSED, pic.PIC_ATTEND_CACHE):
            out = torch.empty((L, 1, H, LATENT), dtype=torch.float32, device=DEV)
            lse = torch.empty((L, 1, H), dtype=torch.float32, device=DEV)
            pic.pic_attend_decode(st.ctx, st.plans, src, q, scale, st.k_pool, None, st.k_cache, None, out, lse, ws)
            assert pic.pic_query_device_status(st.ctx, ws) == 0
            res[src] = (out.cpu().double().numpy(), lse.cpu().double().numpy())
        out, lse = res[pic.PIC_ATTEND_FUSED]
        layers = [0, 30, 60]
        sources = {pic.pic_lookup_chunk(st.ctx, W.chunk_key(wl.name, c)): ("pool", off)
                   for c, off in enumerate(wl.pool_offsets)}
        S = dict(m=m, plans=st.plans, tables=list(st.tables), sources=sources, bs=m.block_size,
                 pool=st.k_pool[layers].cpu(), cache=st.k_cache[layers].cpu())
        rows, segs, T = _context_rows(S, 0)
        assert T == 65536
        qb = bits(q)
        for i, l in enumerate(layers):
            o, s = oracle.attention_decode(oracle.bf16_bits_to_f64(qb[l, 0]), rows[i][:, None, :],
                                           rows[i][:, None, :LATENT], scale, None)
            np.testing.assert_allclose(out[l, 0], o, atol=2e-3, rtol=0)
            np.testing.assert_allclose(lse[l, 0], s, atol=2e-3, rtol=0)
        out_c, lse_c = res[pic.PIC_ATTEND_CACHE]
        np.testing.assert_allclose(out_c, out, atol=3e-2, rtol=0)
        np.testing.assert_allclose(lse_c, lse, atol=3e-2, rtol=0)
    finally:
        st.close()
        torch.cuda.empty_cache()


def test_mla_plan_image_kept_on_device_across_head_counts_and_layer_windows():
    """One context alternates 16 and 32 query heads (the query-rotating and
    the key-rotating tiles, each its own cached plan and device image) and
    two layer windows, on two workspaces: every call must equal the first
    call of the same configuration bit for bit, and that one the oracle."""
    S = _setup("interleaved", 2, seed=6)
    try:
        ctx, L = S["ctx"], S["L"]
        g = torch.Generator().manual_seed(8)
        q_all = torch.randn((L, 3, 32, ROW), generator=g).to(torch.bfloat16).to(DEV)
        scale = 1.0 / math.sqrt(192)
        pool, cache = S["pool"].to(DEV), S["cache"].to(DEV)
        nbytes = max(pic.pic_attend_workspace_bytes(ctx, S["plans"], H, L) for H in (16, 32))
        wss = [torch.full((nbytes,), 0xCD, dtype=torch.uint8, device=DEV) for _ in range(2)]
        first = {}
        order = [(16, 0, 2), (32, 0, 2), (16, 1, 1), (32, 0, 2), (16, 0, 2), (32, 1, 1), (16, 1, 1), (32, 1, 1)]
        for i, (H, lb, nl) in enumerate(order):
            q = q_all[lb:lb + nl, :, :H].contiguous()
            out = torch.full((nl, 3, H, LATENT), float("nan"), dtype=torch.float32, device=DEV)
            lse = torch.full((nl, 3, H), float("nan"), dtype=torch.float32, device=DEV)
            ws = wss[i % 2]
            pic.pic_attend_decode(ctx, S["plans"], pic.PIC_ATTEND_FUSED, q, scale, pool, None, cache, None, out, lse,
                                  ws, sink_bias=-15.0, layer_begin=lb)
            torch.cuda.synchronize()
            assert pic.pic_query_device_status(ctx, ws) == 0, (i, H, lb)
            got = (out.cpu().numpy(), lse.cpu().numpy())
            key = (H, lb, nl)
            if key not in first:
                first[key] = got
            else:
                assert np.array_equal(got[0], first[key][0]) and np.array_equal(got[1], first[key][1]), (i, key)
        for H in (16, 32):
            q = q_all[:, :, :H].cpu()
            out, lse = first[(H, 0, 2)]
            _check_against_oracle(S, q, out.astype(np.float64), lse.astype(np.float64), scale, -15.0, 2e-3)
            out1, _ = first[(H, 1, 1)]
            np.testing.assert_allclose(out1, out[1:2], atol=1e-4, rtol=0)
    finally:
        pic.pic_destroy(S["ctx"])
