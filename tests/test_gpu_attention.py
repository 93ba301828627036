"""GPU parity of decode attention over a stitched context: the fused path
(chunk keys rotated on their way from the pool into registers) against the
fp64 oracle over exactly rotated keys, with and without LegoLink's sink bias;
the paged-cache path over a materialized stitch against the same oracle
(looser: its keys were rounded to bf16 once)."""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import bits
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
        want, want_lse = _oracle(S, bits(q), scale, -15.0)
        np.testing.assert_allclose(out_f, want, atol=2e-3, rtol=0)
        np.testing.assert_allclose(out_c, want, atol=3e-2, rtol=0)
        np.testing.assert_allclose(lse_c, want_lse, atol=3e-2, rtol=0)
        assert np.abs(out_f - want).max() < np.abs(out_c - want).max()   # fusing skips one rounding
    finally:
        pic.pic_destroy(S["ctx"])
