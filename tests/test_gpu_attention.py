"""GPU parity of decode attention over a stitched context: the fused path
(chunk keys rotated on their way from the pool into registers) against the
fp64 oracle over exactly rotated keys, with and without LegoLink's sink bias;
the paged-cache path over a materialized stitch against the oracle over the
stitched bf16 keys it reads (same tolerance), and against the exact-key
oracle (looser: its keys were rounded to bf16 once)."""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import Stitched, bits, random_attend_layout, register_attend_layout
from position_independent_kv_stitch_gb300 import pic

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pic.load(build_if_missing=True)


def _setup(pairing, D, Hkv, G, L, seed=0):
    bs = 16
    m = W.Model("attn", "gqa", L, Hkv, D, D, 0, pairing, 5e5, bs, W.LLAMA3_SCALING)
    lens = [40, 100, 7, 33, 64]
    offs = [0, 40, 140, 147, 180]
    nb = 80
    ctx = pic.create_from_spec(pic.model_spec_from(m), nb)
    for c in range(4):
        pic.pic_register_chunk(ctx, W.chunk_key("attn", c), offs[c], lens[c])
    # chunk 4 lives in cache blocks 70..73 at position 500
    pic.pic_register_chunk_blocks(ctx, W.chunk_key("attn", 4), [70, 71, 72, 73], 64, 500)
    g = torch.Generator().manual_seed(seed)
    shape_pool = (L, 244, Hkv, D)
    k_pool = torch.randn(shape_pool, generator=g).to(torch.bfloat16)
    v_pool = torch.randn(shape_pool, generator=g).to(torch.bfloat16)
    shape_cache = (L, nb, bs, Hkv, D)
    k_cache = torch.randn(shape_cache, generator=g).to(torch.bfloat16)
    v_cache = torch.randn(shape_cache, generator=g).to(torch.bfloat16)
    # request 0: 5 inline tokens, chunks 1, 0, 4 (block-resident, copied), 3, then 9 inline tokens
    # request 1: chunks 2, 3, 1 from position 0
    p0, bt0 = pic.pic_build_block_table(ctx, [1, 0, 4, 3], 20, start_pos=5, total_tokens=5 + 100 + 40 + 64 + 33 + 9,
                                        k_nonleading=4)
    p1, bt1 = pic.pic_build_block_table(ctx, [2, 3, 1], 20, k_nonleading=4)
    return dict(m=m, ctx=ctx, plans=[p0, p1], tables=[bt0, bt1], k_pool=k_pool, v_pool=v_pool, k_cache=k_cache,
                v_cache=v_cache, lens=lens, offs=offs, bs=bs, Hq=Hkv * G, D=D, L=L)


def _oracle(S, q, scale, bias_value):
    """Keys/values of every context position from their sources, exactly rotated."""
    m, bs = S["m"], S["bs"]
    theta = oracle.model_inv_freq(m.rope_dim, m.rope_theta, m.llama3)
    pairing = oracle.NEOX_HALF if m.pairing == "neox" else oracle.INTERLEAVED
    kp, vp = oracle.bf16_bits_to_f64(bits(S["k_pool"])), bits(S["v_pool"])
    kc, vc = oracle.bf16_bits_to_f64(bits(S["k_cache"])), bits(S["v_cache"])
    chunk_specs = [oracle.Chunk(S["offs"][c], S["lens"][c], 0) for c in range(4)]
    outs, lses = [], []
    for r, plan in enumerate(S["plans"]):
        info = pic.pic_plan_info(plan)
        T = info["total_tokens"]
        table = S["tables"][r]
        keys = np.empty((S["L"], T, m.num_kv_heads, m.head_dim))
        vals = np.empty((S["L"], T, m.num_kv_heads, m.head_dim))
        for p in range(T):
            keys[:, p] = kc[:, table[p // bs], p % bs]
            vals[:, p] = oracle.bf16_bits_to_f64(vc[:, table[p // bs], p % bs])
        segs = []
        for j in range(info["num_segments"]):
            sg = pic.pic_plan_segment(plan, j)
            segs.append(oracle.Segment(sg["chunk_id"], sg["src_tok"], sg["num_tokens"], sg["dst_pos"], sg["delta"]))
            for t in range(sg["num_tokens"]):
                p = sg["dst_pos"] + t
                if sg["chunk_id"] < 4:
                    src_k, src_v = kp[:, sg["src_tok"] + t], oracle.bf16_bits_to_f64(vp[:, sg["src_tok"] + t])
                else:
                    blk = [70, 71, 72, 73][t // bs]
                    src_k, src_v = kc[:, blk, t % bs], oracle.bf16_bits_to_f64(vc[:, blk, t % bs])
                keys[:, p] = oracle.rotate(src_k, sg["delta"], theta, pairing)
                vals[:, p] = src_v
        bias = oracle.sink_bias(segs, T, 4, bias_value) if bias_value else None
        o_l, s_l = [], []
        for l in range(S["L"]):
            o, s = oracle.attention_decode(oracle.bf16_bits_to_f64(q[l, r]), keys[l], vals[l], scale, bias)
            o_l.append(o)
            s_l.append(s)
        outs.append(np.stack(o_l))
        lses.append(np.stack(s_l))
    return np.stack(outs, axis=1), np.stack(lses, axis=1)


def _oracle_over_cache(S, k_cache_bits, v_cache_bits, q, scale, bias_value):
    """The oracle's attention over the keys and values as a stitch left them
    in the paged cache (bf16, already rotated): what the cache path reads."""
    m, bs = S["m"], S["bs"]
    kc, vc = oracle.bf16_bits_to_f64(k_cache_bits), oracle.bf16_bits_to_f64(v_cache_bits)
    outs, lses = [], []
    for r, plan in enumerate(S["plans"]):
        info = pic.pic_plan_info(plan)
        T = info["total_tokens"]
        table = S["tables"][r]
        keys = np.stack([kc[:, table[p // bs], p % bs] for p in range(T)], axis=1)
        vals = np.stack([vc[:, table[p // bs], p % bs] for p in range(T)], axis=1)
        segs = []
        for j in range(info["num_segments"]):
            sg = pic.pic_plan_segment(plan, j)
            segs.append(oracle.Segment(sg["chunk_id"], sg["src_tok"], sg["num_tokens"], sg["dst_pos"], sg["delta"]))
        bias = oracle.sink_bias(segs, T, 4, bias_value) if bias_value else None
        o_l, s_l = [], []
        for l in range(S["L"]):
            o, s_ = oracle.attention_decode(oracle.bf16_bits_to_f64(q[l, r]), keys[l], vals[l], scale, bias)
            o_l.append(o)
            s_l.append(s_)
        outs.append(np.stack(o_l))
        lses.append(np.stack(s_l))
    return np.stack(outs, axis=1), np.stack(lses, axis=1)


def _run(S, source, bias_value=0.0, k_cache=None, v_cache=None):
    L, Hq, D = S["L"], S["Hq"], S["D"]
    g = torch.Generator().manual_seed(9)
    q = torch.randn((L, 2, Hq, D), generator=g).to(torch.bfloat16)
    out = torch.empty((L, 2, Hq, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((L, 2, Hq), dtype=torch.float32, device=DEV)
    ws = torch.empty(pic.pic_attend_workspace_bytes(S["ctx"], S["plans"], Hq, L), dtype=torch.uint8, device=DEV)
    scale = 1.0 / math.sqrt(D)
    kc = k_cache if k_cache is not None else S["k_cache"].to(DEV)
    vc = v_cache if v_cache is not None else S["v_cache"].to(DEV)
    pic.pic_attend_decode(S["ctx"], S["plans"], source, q.to(DEV), scale, S["k_pool"].to(DEV), S["v_pool"].to(DEV),
                          kc, vc, out, lse, ws, sink_bias=bias_value)
    torch.cuda.synchronize()
    return q, out.cpu().double().numpy(), lse.cpu().double().numpy(), scale


@pytest.mark.parametrize("pairing,D,Hkv,G", [("neox", 128, 2, 4), ("interleaved", 128, 2, 4), ("neox", 64, 4, 2),
                                             ("neox", 128, 1, 8), ("interleaved", 64, 2, 1)])
@pytest.mark.parametrize("bias_value", [0.0, -15.0])
def test_fused_attention_matches_oracle(pairing, D, Hkv, G, bias_value):
    S = _setup(pairing, D, Hkv, G, 2)
    try:
        q, out, lse, scale = _run(S, pic.PIC_ATTEND_FUSED, bias_value)
        want, want_lse = _oracle(S, bits(q), scale, bias_value)
        np.testing.assert_allclose(out, want, atol=2e-3, rtol=0)
        np.testing.assert_allclose(lse, want_lse, atol=2e-3, rtol=0)
    finally:
        pic.pic_destroy(S["ctx"])


def test_cache_path_over_materialized_stitch():
    """Stitch the two requests into the cache, then attend from the cache:
    the same result up to the one bf16 rounding of the stitched keys."""
    S = _setup("neox", 128, 2, 4, 2)
    try:
        ctx = S["ctx"]
        kc, vc = S["k_cache"].to(DEV), S["v_cache"].to(DEV)
        d_bt = torch.from_numpy(np.stack(S["tables"])).to(DEV)
        ws = torch.empty(pic.pic_workspace_bytes(ctx, S["plans"]), dtype=torch.uint8, device=DEV)
        pic.pic_stitch(ctx, S["plans"], S["k_pool"].to(DEV), S["v_pool"].to(DEV), kc, vc, d_bt, None, None, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0
        q, out_c, lse_c, scale = _run(S, pic.PIC_ATTEND_CACHE, -15.0, kc, vc)
        _, out_f, lse_f, _ = _run(S, pic.PIC_ATTEND_FUSED, -15.0, kc, vc)
        # the cache path against the oracle over the very keys it reads
        # (the GPU-stitched bf16 rows), at the attention tolerance
        want_c, want_c_lse = _oracle_over_cache(S, bits(kc), bits(vc), bits(q), scale, -15.0)
        np.testing.assert_allclose(out_c, want_c, atol=2e-3, rtol=0)
        np.testing.assert_allclose(lse_c, want_c_lse, atol=2e-3, rtol=0)
        # both paths against the oracle over exactly rotated keys: the cache
        # path differs by the one bf16 rounding of its stitched keys
        want, want_lse = _oracle(S, bits(q), scale, -15.0)
        np.testing.assert_allclose(out_f, want, atol=2e-3, rtol=0)
        np.testing.assert_allclose(out_c, want, atol=3e-2, rtol=0)
        np.testing.assert_allclose(lse_c, want_lse, atol=3e-2, rtol=0)
        assert np.abs(out_f - want).max() < np.abs(out_c - want).max()   # fusing skips one rounding
    finally:
        pic.pic_destroy(S["ctx"])


# ---------------------------------------------------------------------------
# long contexts: many stages per key, CTAs spanning several keys and keys
# spread over several CTAs, head groups, every query-group size
# ---------------------------------------------------------------------------

_POOL_LENS = [1, 5, 16, 17, 33, 100, 250, 300, 64, 128, 7, 400]
_BLOCK_CHUNK = (45, [190, 191, 192], 700)   # tokens, blocks, position its keys sit at


def _long_setup(pairing, D, Hkv, G, L, seed, rep=1):
    bs, nb = 16, 200 + 120 * (rep - 1)
    m = W.Model("attn-long", "gqa", L, Hkv, D, D, 0, pairing, 1e6, bs)
    ctx = pic.create_from_spec(pic.model_spec_from(m), nb)
    offs = [0]
    for n in _POOL_LENS[:-1]:
        offs.append(offs[-1] + n)
    ids, sources = [], {}
    for c, (o, n) in enumerate(zip(offs, _POOL_LENS)):
        cid = pic.pic_register_chunk(ctx, W.chunk_key("attn-long", c), o, n)[0]
        ids.append(cid)
        sources[cid] = ("pool", o)
    n_b, blocks, base = _BLOCK_CHUNK
    bid = pic.pic_register_chunk_blocks(ctx, W.chunk_key("attn-long", 99), blocks, n_b, base)[0]
    sources[bid] = ("blocks", blocks)
    g = torch.Generator().manual_seed(seed)
    P = offs[-1] + _POOL_LENS[-1]
    k_pool = torch.randn((L, P, Hkv, D), generator=g).to(torch.bfloat16)
    v_pool = torch.randn((L, P, Hkv, D), generator=g).to(torch.bfloat16)
    k_cache = torch.randn((L, nb, bs, Hkv, D), generator=g).to(torch.bfloat16)
    v_cache = torch.randn((L, nb, bs, Hkv, D), generator=g).to(torch.bfloat16)

    def positions(chunks, start, gaps):
        pos, p = [], start
        for j, c in enumerate(chunks):
            p += gaps.get(j, 0)
            pos.append(p)
            p += n_b if c == bid else _POOL_LENS[ids.index(c)]
        return pos, p

    # rep > 1 repeats each request's pool chunks (a chunk may occur more than
    # once in a request when it is copied) so every CTA owns many stages
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
    return dict(m=m, ctx=ctx, plans=plans, tables=tables, sources=sources, k_pool=k_pool, v_pool=v_pool,
                k_cache=k_cache, v_cache=v_cache, bs=bs, L=L, Hq=Hkv * G, D=D)


def _context_kv(S, r, layers):
    """fp64 keys (exactly rotated) and values of request r's context."""
    m, bs = S["m"], S["bs"]
    theta = oracle.model_inv_freq(m.rope_dim, m.rope_theta, m.llama3)
    pairing = oracle.NEOX_HALF if m.pairing == "neox" else oracle.INTERLEAVED
    plan, table = S["plans"][r], S["tables"][r]
    T = pic.pic_plan_info(plan)["total_tokens"]
    pos = np.arange(T)
    blk_i = torch.as_tensor(np.asarray(table)[pos // bs], dtype=torch.long)
    row_i = torch.as_tensor(pos % bs, dtype=torch.long)
    kc, vc = S["k_cache"][layers], S["v_cache"][layers]
    keys = oracle.bf16_bits_to_f64(bits(kc[:, blk_i, row_i]))
    vals = oracle.bf16_bits_to_f64(bits(vc[:, blk_i, row_i]))
    segs = []
    for j in range(pic.pic_plan_info(plan)["num_segments"]):
        sg = pic.pic_plan_segment(plan, j)
        n, p0 = sg["num_tokens"], sg["dst_pos"]
        kind, where = S["sources"][sg["chunk_id"]]
        t = np.arange(n)
        if kind == "pool":
            src = torch.as_tensor(sg["src_tok"] + t, dtype=torch.long)
            src_k = S["k_pool"][layers][:, src]
            src_v = S["v_pool"][layers][:, src]
        else:   # a block-resident chunk, used from its first token (src_tok is -1 there)
            loc = t
            blk = torch.as_tensor(np.asarray(where)[loc // bs], dtype=torch.long)
            row = torch.as_tensor(loc % bs, dtype=torch.long)
            src_k = S["k_cache"][layers][:, blk, row]
            src_v = S["v_cache"][layers][:, blk, row]
        keys[:, p0:p0 + n] = oracle.rotate(oracle.bf16_bits_to_f64(bits(src_k)), sg["delta"], theta, pairing)
        vals[:, p0:p0 + n] = oracle.bf16_bits_to_f64(bits(src_v))
        segs.append(oracle.Segment(sg["chunk_id"], sg["src_tok"], n, p0, sg["delta"]))
    return keys, vals, segs, T


@pytest.mark.parametrize("pairing,D,Hkv,G,L,bias_value,rep", [
    ("neox", 128, 8, 4, 3, -15.0, 1),
    ("interleaved", 64, 16, 2, 2, 0.0, 1),
    ("neox", 64, 8, 8, 2, -15.0, 1),
    ("neox", 128, 8, 8, 2, 0.0, 1),
    ("interleaved", 128, 2, 1, 2, -15.0, 1),
    ("neox", 128, 8, 4, 3, -15.0, 6),
    ("neox", 64, 8, 8, 2, 0.0, 4),
    ("interleaved", 128, 2, 1, 2, -15.0, 4),
    ("interleaved", 64, 16, 2, 2, -15.0, 4),
])
def test_fused_attention_long_mixed_contexts(pairing, D, Hkv, G, L, bias_value, rep):
    """Three requests of 250-1,400 positions (times rep): chunks of 1..400
    tokens (so stages of every length and delta changes inside a CTA's
    range), inline gaps and a trailing run of inline tokens, a block-resident
    chunk read from its blocks; every (layer, request, query head) against
    the oracle.  With rep > 1 every CTA owns many more stages than its ring
    has slots, so slots are refilled while the others are in flight."""
    S = _long_setup(pairing, D, Hkv, G, L, seed=4, rep=rep)
    try:
        layers = list(range(L))
        g = torch.Generator().manual_seed(5)
        q = torch.randn((L, 3, S["Hq"], D), generator=g).to(torch.bfloat16)
        out = torch.empty((L, 3, S["Hq"], D), dtype=torch.float32, device=DEV)
        lse = torch.empty((L, 3, S["Hq"]), dtype=torch.float32, device=DEV)
        ws = torch.empty(pic.pic_attend_workspace_bytes(S["ctx"], S["plans"], S["Hq"], L), dtype=torch.uint8,
                         device=DEV)
        scale = 1.0 / math.sqrt(D)
        pic.pic_attend_decode(S["ctx"], S["plans"], pic.PIC_ATTEND_FUSED, q.to(DEV), scale, S["k_pool"].to(DEV),
                              S["v_pool"].to(DEV), S["k_cache"].to(DEV), S["v_cache"].to(DEV), out, lse, ws,
                              sink_bias=bias_value)
        assert pic.pic_query_device_status(S["ctx"], ws) == 0
        out, lse = out.cpu().double().numpy(), lse.cpu().double().numpy()
        qb = bits(q)
        for r in range(3):
            keys, vals, segs, T = _context_kv(S, r, layers)
            bias = oracle.sink_bias(segs, T, 4, bias_value) if bias_value else None
            for l in layers:
                o, s = oracle.attention_decode(oracle.bf16_bits_to_f64(qb[l, r]), keys[l], vals[l], scale, bias)
                np.testing.assert_allclose(out[l, r], o, atol=2e-3, rtol=0)
                np.testing.assert_allclose(lse[l, r], s, atol=2e-3, rtol=0)
    finally:
        pic.pic_destroy(S["ctx"])


def _random_setup(seed):
    """A seeded random GQA context: either pairing, head_dim 64 or 128, 1-16
    KV heads (3 and 5 included, 16 as two head groups), 1-8 query heads per
    KV head, 1-3 layers, block size 1-33, plain or Llama-3.1 frequencies, and
    the chunk and request mix of random_attend_layout."""
    rng = np.random.default_rng(3000 + seed)
    pairing = ["neox", "interleaved"][int(rng.integers(2))]
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 3, 5, 8, 16]))
    G = int(rng.choice([1, 2, 4, 8]))
    L = int(rng.integers(1, 4))
    bs = int(rng.choice([1, 4, 16, 33]))
    theta = float(rng.choice([1e4, 5e5, 1e6]))
    m = W.Model(f"attn-rand-{seed}", "gqa", L, Hkv, D, D, 0, pairing, theta, bs,
                W.LLAMA3_SCALING if rng.random() < 0.3 else None)
    lay = random_attend_layout(rng, bs)
    ctx = pic.create_from_spec(pic.model_spec_from(m), lay["nb"])
    plans, tables, sources = register_attend_layout(ctx, lay, m.name, bs)
    g = torch.Generator().manual_seed(seed)
    k_pool = torch.randn((L, lay["P"], Hkv, D), generator=g).to(torch.bfloat16)
    v_pool = torch.randn((L, lay["P"], Hkv, D), generator=g).to(torch.bfloat16)
    k_cache = torch.randn((L, lay["nb"], bs, Hkv, D), generator=g).to(torch.bfloat16)
    v_cache = torch.randn((L, lay["nb"], bs, Hkv, D), generator=g).to(torch.bfloat16)
    return dict(m=m, ctx=ctx, plans=plans, tables=tables, sources=sources, k_pool=k_pool, v_pool=v_pool,
                k_cache=k_cache, v_cache=v_cache, bs=bs, L=L, Hq=Hkv * G, D=D, k=lay["k"], rng=rng)


@pytest.mark.parametrize("seed", range(10))
def test_random_contexts_match_oracle(seed):
    """Seeded random contexts (geometry, chunk lengths, block-resident chunks,
    repeats, truncation, inline gaps, pseudo-sink widths, a random layer
    window), both sources: fused against the oracle over exactly rotated
    keys, the cache path against the oracle over the cache rows as stored;
    every (layer, request, query head) within 2e-3."""
    S = _random_setup(seed)
    try:
        rng, ctx, plans = S["rng"], S["ctx"], S["plans"]
        L, Hq, D, n = S["L"], S["Hq"], S["D"], len(plans)
        bias_value = -15.0 if rng.random() < 0.5 else 0.0
        lb = int(rng.integers(0, L))
        nl = int(rng.integers(1, L - lb + 1))
        layers = list(range(lb, lb + nl))
        q = torch.randn((nl, n, Hq, D), generator=torch.Generator().manual_seed(50 + seed)).to(torch.bfloat16)
        qb = bits(q)
        scale = 1.0 / math.sqrt(D)
        dev = {k: S[k].to(DEV) for k in ("k_pool", "v_pool", "k_cache", "v_cache")}
        ws = torch.empty(pic.pic_attend_workspace_bytes(ctx, plans, Hq, nl), dtype=torch.uint8, device=DEV)
        bs = S["bs"]
        for source in (pic.PIC_ATTEND_FUSED, pic.PIC_ATTEND_CACHE):
            out = torch.full((nl, n, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
            lse = torch.full((nl, n, Hq), float("nan"), dtype=torch.float32, device=DEV)
            pic.pic_attend_decode(ctx, plans, source, q.to(DEV), scale, dev["k_pool"], dev["v_pool"], dev["k_cache"],
                                  dev["v_cache"], out, lse, ws, sink_bias=bias_value, layer_begin=lb)
            assert pic.pic_query_device_status(ctx, ws) == 0
            out, lse = out.cpu().double().numpy(), lse.cpu().double().numpy()
            for r in range(n):
                keys, vals, segs, T = _context_kv(S, r, layers)
                if source == pic.PIC_ATTEND_CACHE:
                    pos = np.arange(T)
                    table = np.asarray(S["tables"][r])
                    keys = oracle.bf16_bits_to_f64(bits(S["k_cache"][layers]))[:, table[pos // bs], pos % bs]
                    vals = oracle.bf16_bits_to_f64(bits(S["v_cache"][layers]))[:, table[pos // bs], pos % bs]
                bias = oracle.sink_bias(segs, T, S["k"], bias_value) if bias_value else None
                for i in range(nl):
                    o, s_ = oracle.attention_decode(oracle.bf16_bits_to_f64(qb[i, r]), keys[i], vals[i], scale, bias)
                    np.testing.assert_allclose(out[i, r], o, atol=2e-3, rtol=0, err_msg=f"source {source} r {r} l {i}")
                    np.testing.assert_allclose(lse[i, r], s_, atol=2e-3, rtol=0, err_msg=f"source {source} r {r} l {i}")
    finally:
        pic.pic_destroy(S["ctx"])


def test_llama_full_launch_sampled_layers():
    """The benchmark's launch (Llama-3.1-8B shapes, 32 layers, 32 query heads,
    10,368 positions, sink bias -15) in one call; layers 0, 17 and 31 against
    the oracle, and the cache path over the stitched copy against the fused
    result everywhere."""
    wl = W.llama31_8b_rag()
    st = Stitched(wl).run()
    try:
        m = wl.model
        Hq, L = 32, m.num_layers
        g = torch.Generator(device=DEV)
        g.manual_seed(11)
        q = torch.empty((L, 1, Hq, 128), dtype=torch.bfloat16, device=DEV).normal_(0.0, 1.0, generator=g)
        scale = 1.0 / math.sqrt(128)
        ws = torch.empty(pic.pic_attend_workspace_bytes(st.ctx, st.plans, Hq, L), dtype=torch.uint8, device=DEV)
        res = {}
        for src in (pic.PIC_ATTEND_FUSED, pic.PIC_ATTEND_CACHE):
            out = torch.empty((L, 1, Hq, 128), dtype=torch.float32, device=DEV)
            lse = torch.empty((L, 1, Hq), dtype=torch.float32, device=DEV)
            pic.pic_attend_decode(st.ctx, st.plans, src, q, scale, st.k_pool, st.v_pool, st.k_cache, st.v_cache,
                                  out, lse, ws, sink_bias=-15.0)
            assert pic.pic_query_device_status(st.ctx, ws) == 0
            res[src] = (out.cpu().double().numpy(), lse.cpu().double().numpy())
        out, lse = res[pic.PIC_ATTEND_FUSED]
        layers = [0, 17, 31]
        sources = {}
        for c, off in enumerate(wl.pool_offsets):
            sources[pic.pic_lookup_chunk(st.ctx, W.chunk_key(wl.name, c))] = ("pool", off)
        S = dict(m=m, plans=st.plans, tables=st.tables, sources=sources, bs=m.block_size,
                 k_pool=st.k_pool[layers].cpu(), v_pool=st.v_pool[layers].cpu(),
                 k_cache=st.k_cache[layers].cpu(), v_cache=st.v_cache[layers].cpu())
        keys, vals, segs, T = _context_kv(S, 0, list(range(len(layers))))
        assert T == 10368
        bias = oracle.sink_bias(segs, T, 4, -15.0)
        qb = bits(q)
        for i, l in enumerate(layers):
            o, s = oracle.attention_decode(oracle.bf16_bits_to_f64(qb[l, 0]), keys[i], vals[i], scale, bias)
            np.testing.assert_allclose(out[l, 0], o, atol=2e-3, rtol=0)
            np.testing.assert_allclose(lse[l, 0], s, atol=2e-3, rtol=0)
        out_c, lse_c = res[pic.PIC_ATTEND_CACHE]
        np.testing.assert_allclose(out_c, out, atol=3e-2, rtol=0)
        np.testing.assert_allclose(lse_c, lse, atol=3e-2, rtol=0)
    finally:
        st.close()
        torch.cuda.empty_cache()


def test_plan_image_kept_on_device_follows_plans_layers_and_workspaces():
    """The context keeps each cached attention plan's read-only image (stages,
    token rows, record keys) on the device and uploads it again only when the
    plans, the layer count or the grid change; each call zeroes its own
    workspace's status word.  One context alternates two plan sets, two layer
    windows, two workspaces and two streams: every call must equal the first
    call of the same configuration bit for bit, and that one the oracle."""
    S = _setup("neox", 128, 2, 4, 2)
    try:
        ctx, L, Hq, D = S["ctx"], S["L"], S["Hq"], S["D"]
        g = torch.Generator().manual_seed(5)
        q = torch.randn((L, 2, Hq, D), generator=g).to(torch.bfloat16).to(DEV)
        scale = 1.0 / math.sqrt(D)
        kp, vp = S["k_pool"].to(DEV), S["v_pool"].to(DEV)
        kc, vc = S["k_cache"].to(DEV), S["v_cache"].to(DEV)
        nbytes = pic.pic_attend_workspace_bytes(ctx, S["plans"], Hq, L)
        wss = [torch.full((nbytes,), 0xAB, dtype=torch.uint8, device=DEV) for _ in range(2)]
        side = torch.cuda.Stream()
        cases = {
            "both": (S["plans"], slice(0, 2), 0, L),
            "second": ([S["plans"][1]], slice(1, 2), 0, L),
            "both, layer 1": (S["plans"], slice(0, 2), 1, 1),
        }
        first = {}
        order = ["both", "second", "both", "both, layer 1", "second", "both, layer 1", "both", "second"]
        for i, name in enumerate(order):
            plans, rq, lb, nl = cases[name]
            qq = q[lb:lb + nl, rq].contiguous()
            out = torch.full((nl, len(plans), Hq, D), float("nan"), dtype=torch.float32, device=DEV)
            lse = torch.full((nl, len(plans), Hq), float("nan"), dtype=torch.float32, device=DEV)
            ws = wss[i % 2]
            stream = side if i % 3 == 2 else None
            if stream is not None:
                side.wait_stream(torch.cuda.current_stream())
            pic.pic_attend_decode(ctx, plans, pic.PIC_ATTEND_FUSED, qq, scale, kp, vp, kc, vc, out, lse, ws,
                                  sink_bias=-15.0, layer_begin=lb, stream=stream)
            torch.cuda.synchronize()
            assert pic.pic_query_device_status(ctx, ws) == 0, (i, name)
            got = (out.cpu().numpy(), lse.cpu().numpy())
            if name not in first:
                first[name] = got
            else:
                assert np.array_equal(got[0], first[name][0]) and np.array_equal(got[1], first[name][1]), (i, name)
        want, want_lse = _oracle(S, bits(q.cpu()), scale, -15.0)
        out, lse = first["both"]
        np.testing.assert_allclose(out, want, atol=2e-3, rtol=0)
        np.testing.assert_allclose(lse, want_lse, atol=2e-3, rtol=0)
        out, lse = first["both, layer 1"]
        np.testing.assert_allclose(out, want[1:2], atol=2e-3, rtol=0)
        out, lse = first["second"]
        np.testing.assert_allclose(out, want[:, 1:2], atol=2e-3, rtol=0)
    finally:
        pic.pic_destroy(S["ctx"])
