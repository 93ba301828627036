"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Keys: per element |gpu - oracle| <= 2^-7 |oracle| + 1e-3 (rotation computed
in fp32 and rounded once to bf16).  Values, MLA latents, block tables and
recompute lists: bit-exact.  Destinations are pre-filled with a NaN sentinel
so rows written where nothing belongs, or left unwritten, are caught."""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import (Stitched, assert_k_close, bits, f64, oracle_side, pairing_of, rel_l2,
                      sentinel_like, theta_of)
from position_independent_kv_stitch_gb300 import pic

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pic.load(build_if_missing=True)
    yield
    torch.cuda.empty_cache()


@pytest.fixture(params=["bulk", "regs"])
def variant(request, monkeypatch):
    """Runs a test once per kernel variant, forced at pic_create through PIC_KERNEL
    (the default picks the bulk pipeline for MLA rows, registers for GQA rows)."""
    monkeypatch.setenv("PIC_KERNEL", request.param)
    return request.param


def _pairs_close(got, want, pairing, rel, abs_=1e-3):
    a, b = oracle.rope_pairs(want.shape[-1], pairing)
    err = np.hypot(got[..., a] - want[..., a], got[..., b] - want[..., b])
    norm = np.hypot(want[..., a], want[..., b])
    return bool(np.all(err <= rel * norm + abs_)), float(err.max())


# ------------------------------------------------------------- angle probe

@pytest.mark.parametrize("rope_dim,base,llama3", [(128, 5e5, W.LLAMA3_SCALING), (128, 1e6, None),
                                                  (64, 1e4, None)])
def test_cossin_matches_fp64(rope_dim, base, llama3):
    """The kernels' cos/sin of delta*theta_i for every delta in [-2^17, 2^17]
    and a sample up to 2^24 - 1, against float64."""
    kind = pic.PIC_KIND_GQA if rope_dim == 128 else pic.PIC_KIND_MLA
    args = (kind, 1, 8, 128, 128, 0) if kind == pic.PIC_KIND_GQA else (kind, 1, 1, 576, 64, 512)
    ctx = pic.pic_create(*args, pic.PIC_PAIRING_NEOX_HALF, 16, base, 4, llama3=llama3)
    try:
        theta = oracle.model_inv_freq(rope_dim, base, llama3)
        rng = np.random.default_rng(0)
        extra = rng.integers(-(2 ** 24) + 1, 2 ** 24, size=1 << 16)
        deltas = np.concatenate([np.arange(-(2 ** 17), 2 ** 17 + 1), extra, [2 ** 24 - 1, -(2 ** 24) + 1]])
        d = torch.from_numpy(deltas.astype(np.int32)).to(DEV)
        out = torch.empty((len(deltas), rope_dim // 2, 2), dtype=torch.float32, device=DEV)
        ws = torch.empty(4096, dtype=torch.uint8, device=DEV)
        pic.pic_rotation_cossin(ctx, d, out, ws)
        got = out.cpu().double().numpy()
        phi = deltas[:, None].astype(np.float64) * theta[None, :]
        err = max(np.abs(got[..., 0] - np.cos(phi)).max(), np.abs(got[..., 1] - np.sin(phi)).max())
        assert err < 1e-6, err
    finally:
        pic.pic_destroy(ctx)


def _library_theta(ctx, half):
    """The frequencies the kernels use, read back through
    pic_rotation_cossin: each theta_i is refined over shifts 1, 2, 4, ...
    up to the last one that turns it by less than 3 radians (no wrap), so
    the angle error of about 1e-6 is at most 1e-6 relative."""
    deltas = np.array([1 << k for k in range(24)], dtype=np.int32)
    out = torch.empty((len(deltas), half, 2), dtype=torch.float32, device=DEV)
    ws = torch.empty(4096, dtype=torch.uint8, device=DEV)
    pic.pic_rotation_cossin(ctx, torch.from_numpy(deltas).to(DEV), out, ws)
    o = out.cpu().double().numpy()
    ang = np.arctan2(o[..., 1], o[..., 0])
    theta = ang[0].copy()                      # shift 1: theta_i <= 1 < pi
    for k in range(1, len(deltas)):
        grow = theta * deltas[k] < 3.0
        theta[grow] = ang[k][grow] / deltas[k]
    return theta


def test_library_llama3_table_hand_derived():
    """The library's own Llama-3.1 rescaling, tied to hand-derived values
    rather than to the oracle: (1) Llama-3.1-8B's table keeps frequencies
    0-28, divides 35-63 by 8 and blends 29-34 strictly between; (2) one
    frequency placed by the choice of base at each hand-picked wavelength
    (test_oracle_rope.LLAMA3_HAND: s = 0, 1/4, 1/2, 3/4, 1 and both outer
    regimes) comes out at the hand-derived ratio; (3) factor 1 changes
    nothing."""
    from test_oracle_rope import LLAMA3_HAND
    ctx = pic.pic_create(pic.PIC_KIND_GQA, 1, 8, 128, 128, 0, pic.PIC_PAIRING_NEOX_HALF, 16, 5e5, 4,
                         llama3=W.LLAMA3_SCALING)
    try:
        r = _library_theta(ctx, 64) / oracle.rope_inv_freq(128, 5e5)
    finally:
        pic.pic_destroy(ctx)
    np.testing.assert_allclose(r[:29], 1.0, rtol=1e-5)
    np.testing.assert_allclose(r[35:], 0.125, rtol=1e-5)
    assert np.all((r[29:35] > 0.13) & (r[29:35] < 0.99))

    for lam, ratio in LLAMA3_HAND:
        # head_dim 64: theta_16 = b^(-1/2), so b = (lambda / 2 pi)^2 puts
        # frequency 16 at wavelength lambda
        b = (lam / (2 * math.pi)) ** 2
        ctx = pic.pic_create(pic.PIC_KIND_GQA, 1, 1, 64, 64, 0, pic.PIC_PAIRING_NEOX_HALF, 16, b, 4,
                             llama3=W.LLAMA3_SCALING)
        try:
            th16 = _library_theta(ctx, 32)[16]
        finally:
            pic.pic_destroy(ctx)
        assert abs(th16 / (2 * math.pi / lam) - ratio) <= 1e-5 * ratio, (lam, th16 / (2 * math.pi / lam), ratio)

    one = dict(W.LLAMA3_SCALING, factor=1.0)
    ctx = pic.pic_create(pic.PIC_KIND_GQA, 1, 8, 128, 128, 0, pic.PIC_PAIRING_NEOX_HALF, 16, 5e5, 4, llama3=one)
    try:
        np.testing.assert_allclose(_library_theta(ctx, 64) / oracle.rope_inv_freq(128, 5e5), 1.0, rtol=1e-5)
    finally:
        pic.pic_destroy(ctx)


# --------------------------------------------------------- full comparisons

def test_tiny_gqa_full_parity(variant):
    wl = W.tiny_gqa()
    st = Stitched(wl, pool_device="cpu").run()
    try:
        assert pic.pic_kernel_variant(st.ctx, 0) == (pic.PIC_VARIANT_BULK_PIPELINE if variant == "bulk"
                                                      else pic.PIC_VARIANT_REGISTERS)
        segs, tables, rec = oracle_side(wl, st.nb)
        assert st.tables[0][:len(tables[0])].tolist() == tables[0]
        want_k, want_v = oracle.stitch_paged(bits(st.k_pool), bits(st.v_pool), segs, tables, st.nb,
                                             st.bs, theta_of(wl.model), pairing_of(wl.model), 0, 128)
        got_k = f64(st.k_cache)
        assert_k_close(got_k, want_k, "K")
        assert rel_l2(got_k, want_k) <= 4.7e-3  # Irminsul's bf16 delta-rotation error, section 3
        np.testing.assert_array_equal(bits(st.v_cache), want_v)
        assert np.all(bits(st.k_cache)[np.isnan(want_k)] == 0xFFFF)
        indptr, idx = oracle.recompute_csr(rec)
        assert st.indptr.cpu().tolist() == indptr.tolist()
        assert st.ridx.cpu().numpy()[:st.n_rec].tolist() == idx.tolist()
        assert st.n_rec == 16
    finally:
        st.close()


def _custom_workload(name, kind, L, H, D, pairing, bs, lens, requests, theta=1e4, k=(4, 0)):
    if kind == "gqa":
        m = W.Model(name, "gqa", L, H, D, D, 0, pairing, theta, bs)
    else:
        m = W.Model(name, "mla", L, 1, 576, 64, 512, pairing, theta, bs)
    return W.Workload(name, m, lens, requests, k[0], k[1])


GEOMS = [
    ("neox", 128, 8, 16), ("interleaved", 128, 8, 16), ("neox", 64, 3, 5), ("interleaved", 64, 1, 1),
    ("neox", 256, 2, 32), ("interleaved", 256, 4, 7), ("neox", 128, 1, 256),
]


@pytest.mark.parametrize("pairing,D,H,bs", GEOMS)
def test_gqa_geometries_ragged(pairing, D, H, bs, variant):
    """Ragged chunks (1, 15, 17, 33, 100 tokens), a truncated chunk, a repeated
    chunk, two requests in one launch, 3 layers."""
    lens = [1, 15, 17, 33, 100, 64]
    reqs = [[(4, 100), (0, 1), (2, 17), (1, 15), (4, 40)], [(3, 33), (5, 0), (2, 17), (0, 1)]]
    wl = _custom_workload(f"geom-{pairing}-{D}-{H}-{bs}", "gqa", 3, H, D, pairing, bs, lens, reqs)
    st = Stitched(wl, pool_device="cpu", spare_blocks=3).run()
    try:
        segs, tables, rec = oracle_side(wl, st.nb)
        for r in range(2):
            assert st.tables[r][:len(tables[r])].tolist() == tables[r]
        want_k, want_v = oracle.stitch_paged(bits(st.k_pool), bits(st.v_pool), segs, tables, st.nb,
                                             bs, theta_of(wl.model), pairing_of(wl.model), 0, D)
        assert_k_close(f64(st.k_cache), want_k, "K")
        np.testing.assert_array_equal(bits(st.v_cache), want_v)
        assert np.all(bits(st.k_cache)[np.isnan(want_k)] == 0xFFFF)
        indptr, idx = oracle.recompute_csr(rec)
        assert st.indptr.cpu().tolist() == indptr.tolist()
        assert st.ridx.cpu().numpy()[:st.n_rec].tolist() == idx.tolist()
    finally:
        st.close()


def _random_workload(seed):
    """A seeded small batch: GQA or MLA, either pairing, 1-4 layers, odd head
    counts and block sizes, 2-9 chunks of 1-150 tokens, 1-3 requests that
    truncate and repeat chunks, k of 0-6 and a leading carve-out of 0-8."""
    rng = np.random.default_rng(1000 + seed)
    kind = "gqa" if seed % 3 else "mla"
    pairing = ["neox", "interleaved"][int(rng.integers(2))]
    L = int(rng.integers(1, 5))
    H = int(rng.choice([1, 2, 3, 8]))
    D = int(rng.choice([64, 128, 256]))
    bs = int(rng.choice([1, 5, 8, 16, 33]))
    lens = [int(x) for x in rng.integers(1, 151, size=int(rng.integers(2, 10)))]
    reqs = []
    for _ in range(int(rng.integers(1, 4))):
        req = []
        for _ in range(int(rng.integers(1, 7))):
            c = int(rng.integers(len(lens)))
            take = lens[c] if rng.random() < 0.7 else int(rng.integers(0, lens[c] + 1))
            req.append((c, take))
        if sum(t for _, t in req) == 0:
            req[0] = (req[0][0], lens[req[0][0]])
        reqs.append(req)
    k = (int(rng.integers(0, 7)), int(rng.integers(0, 9)))
    return _custom_workload(f"rand-{seed}", kind, L, H, D, pairing, bs, lens, reqs,
                            theta=float(rng.choice([1e4, 5e5, 1e6])), k=k)


@pytest.mark.parametrize("seed", range(12))
def test_random_small_batches_match_oracle(seed, variant):
    """Seeded random batches (geometry, chunk lengths, truncation, repeats,
    recompute widths) against the oracle: K within the contract tolerance, V
    and the MLA latent bit for bit, untouched rows left as they were, block
    tables and recompute lists exact."""
    wl = _random_workload(seed)
    m = wl.model
    st = Stitched(wl, pool_device="cpu", spare_blocks=2).run()
    try:
        segs, tables, rec = oracle_side(wl, st.nb)
        for r in range(len(tables)):
            assert st.tables[r][:len(tables[r])].tolist() == tables[r]
        want_k, want_v = oracle.stitch_paged(bits(st.k_pool), None if st.v_pool is None else bits(st.v_pool), segs,
                                             tables, st.nb, st.bs, theta_of(m), pairing_of(m), m.rope_offset,
                                             m.rope_dim)
        got = f64(st.k_cache)
        if m.kind == "gqa":
            assert_k_close(got, want_k, "K")
            np.testing.assert_array_equal(bits(st.v_cache), want_v)
        else:
            written = ~np.isnan(want_k[..., 0])
            wb = np.where(np.isnan(want_k), 0, want_k)
            assert np.array_equal(got[..., :512][written], wb[..., :512][written])
            assert_k_close(got[..., 512:], want_k[..., 512:], "k_r")
        assert np.all(bits(st.k_cache)[np.isnan(want_k)] == 0xFFFF)
        indptr, idx = oracle.recompute_csr(rec)
        assert st.indptr.cpu().tolist() == indptr.tolist()
        assert st.ridx.cpu().numpy()[:st.n_rec].tolist() == idx.tolist()
    finally:
        st.close()


def test_explicit_positions_base_pos_and_extreme_delta(variant):
    """Chunks cached at a non-zero base position (negative delta up to
    -(2^24 - 4)), explicit positions with inline gaps, a delta-0 chunk (bit
    copy), start after an inline prefix."""
    D, H, bs, L = 128, 2, 16, 2
    m = W.Model("edge", "gqa", L, H, D, D, 0, "neox", 5e5, bs, W.LLAMA3_SCALING)
    lens, bases = [40, 23, 7, 16], [0, 2 ** 24 - 1, 1000, 77]
    offs = [0, 40, 63, 70]
    P = 86
    nb = 20
    ctx = pic.create_from_spec(pic.model_spec_from(m), nb)
    try:
        for c in range(4):
            pic.pic_register_chunk(ctx, W.chunk_key("edge", c), offs[c], lens[c], bases[c])
        dst = [3, 50, 77, 200]
        plan, bt = pic.pic_build_block_table(ctx, [0, 1, 3, 2], 16, dst_pos=dst, total_tokens=230,
                                             k_nonleading=4, take_tokens=[40, 23, 16, 7])
        # chunk 3 (base 77) at 77: delta 0; chunk 1 at 50: delta 50 - (2^24 - 1)
        assert pic.pic_plan_segment(plan, 2)["delta"] == 0
        g = torch.Generator().manual_seed(5)
        k_pool = torch.randn((L, P, H, D), generator=g).to(torch.bfloat16)
        v_pool = torch.randn((L, P, H, D), generator=g).to(torch.bfloat16)
        k_cache = sentinel_like((L, nb, bs, H, D), DEV)
        v_cache = sentinel_like((L, nb, bs, H, D), DEV)
        ridx = torch.empty(16, dtype=torch.int32, device=DEV)
        indptr = torch.empty(2, dtype=torch.int32, device=DEV)
        ws = torch.empty(pic.pic_workspace_bytes(ctx, [plan]), dtype=torch.uint8, device=DEV)
        pic.pic_stitch(ctx, [plan], k_pool.to(DEV), v_pool.to(DEV), k_cache, v_cache,
                       torch.from_numpy(bt).to(DEV).view(1, -1), ridx, indptr, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0

        chunks = [oracle.Chunk(offs[c], lens[c], bases[c]) for c in range(4)]
        segs = oracle.compose(chunks, [0, 1, 3, 2], take=[40, 23, 16, 7], dst_pos=dst)
        assert segs[1].delta == 50 - (2 ** 24 - 1)
        o_bt = oracle.BlockPool(nb).allocate(oracle.blocks_needed(230, bs))
        assert bt[:len(o_bt)].tolist() == o_bt
        want_k, want_v = oracle.stitch_paged(bits(k_pool), bits(v_pool), [segs], [o_bt], nb, bs,
                                             theta_of(m), oracle.NEOX_HALF, 0, D)
        got_k = f64(k_cache)
        assert_k_close(got_k, want_k, "K")
        np.testing.assert_array_equal(bits(v_cache), want_v)
        # delta 0 is a pure bit copy
        s = segs[2]
        for t in range(s.length):
            p = s.dst_pos + t
            assert np.array_equal(bits(k_cache[:, o_bt[p // bs], p % bs]), bits(k_pool[:, s.src_tok + t]))
        assert np.all(bits(k_cache)[np.isnan(want_k)] == 0xFFFF)
        rec = oracle.recompute_positions(segs, 4, 0)
        assert ridx.cpu().numpy()[:len(rec)].tolist() == rec and indptr.cpu().tolist() == [0, len(rec)]
    finally:
        pic.pic_destroy(ctx)


def test_empty_batch_and_empty_request(variant):
    m = W.Model("empty", "gqa", 2, 2, 64, 64, 0, "neox", 1e4, 16)
    ctx = pic.create_from_spec(pic.model_spec_from(m), 8)
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("e", 0), 0, 5)
        k_pool = torch.zeros((2, 5, 2, 64), dtype=torch.bfloat16, device=DEV)
        k_cache = sentinel_like((2, 8, 16, 2, 64), DEV)
        v_cache = sentinel_like((2, 8, 16, 2, 64), DEV)
        bt = torch.full((1, 4), -1, dtype=torch.int32, device=DEV)
        ridx = torch.full((4,), -7, dtype=torch.int32, device=DEV)
        indptr = torch.full((3,), -7, dtype=torch.int32, device=DEV)
        # n_req = 0: only indptr[0] = 0 is written
        ws = torch.empty(max(256, pic.pic_workspace_bytes(ctx, [])), dtype=torch.uint8, device=DEV)
        pic.pic_stitch(ctx, [], k_pool, k_pool, k_cache, v_cache, bt, ridx, indptr, ws)
        torch.cuda.synchronize()
        assert indptr.cpu().tolist()[:1] == [0]
        # a request with no chunks and a zero-length take
        p0, b0 = pic.pic_build_block_table(ctx, [], 4)
        p1, b1 = pic.pic_build_block_table(ctx, [0], 4, take_tokens=[0], start_pos=3, k_nonleading=4)
        assert b0.tolist() == [-1] * 4 and pic.pic_plan_info(p1)["num_blocks"] == 1
        bt = torch.from_numpy(np.stack([b0, b1])).to(DEV)
        ws = torch.empty(pic.pic_workspace_bytes(ctx, [p0, p1]), dtype=torch.uint8, device=DEV)
        pic.pic_stitch(ctx, [p0, p1], k_pool, k_pool, k_cache, v_cache, bt, ridx, indptr, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0
        assert indptr.cpu().tolist() == [0, 0, 0]
        assert np.all(bits(k_cache) == 0xFFFF) and np.all(bits(v_cache) == 0xFFFF)
    finally:
        pic.pic_destroy(ctx)


def test_bad_block_entry_sets_status_and_skips_write(variant):
    """A block-table entry outside the cache is caught by the kernel's own
    bounds check: the write is skipped and the status word raised."""
    m = W.Model("bad", "gqa", 1, 1, 64, 64, 0, "neox", 1e4, 16)
    ctx = pic.create_from_spec(pic.model_spec_from(m), 4)
    try:
        pic.pic_register_chunk(ctx, W.chunk_key("b", 0), 0, 20)
        plan, bt = pic.pic_build_block_table(ctx, [0], 2)
        bt[1] = 4  # outside [0, 4)
        k_pool = torch.ones((1, 20, 1, 64), dtype=torch.bfloat16, device=DEV)
        k_cache = sentinel_like((1, 4, 16, 1, 64), DEV)
        v_cache = sentinel_like((1, 4, 16, 1, 64), DEV)
        ws = torch.empty(pic.pic_workspace_bytes(ctx, [plan]), dtype=torch.uint8, device=DEV)
        pic.pic_stitch(ctx, [plan], k_pool, k_pool, k_cache, v_cache,
                       torch.from_numpy(bt).to(DEV).view(1, -1), None, None, ws)
        with pytest.raises(pic.PicError) as e:
            pic.pic_query_device_status(ctx, ws)
        assert e.value.status_name == "PIC_ERR_DEVICE_CHECK"
        kb = bits(k_cache)
        assert np.all(kb[0, 0] == 0x3F80)                 # block 0 written (ones)
        assert np.all(kb[0, 1:] == 0xFFFF)                # nothing else touched
    finally:
        pic.pic_destroy(ctx)


def test_llama31_8b_full_parity_on_three_layers():
    """Llama-3.1-8B shapes (32 layers, llama3-scaled theta 5e5): the whole
    launch as the benchmark runs it; layers 0, 13 and 31 compared in full."""
    wl = W.llama31_8b_rag()
    st = Stitched(wl).run()
    try:
        segs, tables, rec = oracle_side(wl, st.nb)
        assert st.tables[0][:len(tables[0])].tolist() == tables[0]
        layers = [0, 13, 31]
        kp = bits(st.k_pool[layers])
        vp = bits(st.v_pool[layers])
        want_k, want_v = oracle.stitch_paged(kp, vp, segs, tables, st.nb, st.bs, theta_of(wl.model),
                                             pairing_of(wl.model), 0, 128)
        got_k = f64(st.k_cache[layers])
        assert_k_close(got_k, want_k, "K")
        assert rel_l2(got_k, want_k) <= 4.7e-3
        np.testing.assert_array_equal(bits(st.v_cache[layers]), want_v)
        # every layer's V equals the pool gathered by the oracle's table (bit copy)
        flat_src = np.concatenate([np.arange(s.src_tok, s.src_tok + s.length) for s in segs[0]])
        pos = np.concatenate([np.arange(s.dst_pos, s.dst_pos + s.length) for s in segs[0]])
        blk = torch.as_tensor(np.asarray(tables[0])[pos // 16], device=DEV)
        row = torch.as_tensor(pos % 16, device=DEV)
        src = torch.as_tensor(flat_src, device=DEV)
        for l in range(wl.model.num_layers):
            assert torch.equal(st.v_cache[l, blk, row].view(torch.int16), st.v_pool[l, src].view(torch.int16))
        assert st.ridx.cpu().numpy()[:st.n_rec].tolist() == rec[0] and st.n_rec == 40
    finally:
        st.close()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("pairing", ["interleaved", "neox"])
def test_mla_parity_small_context(pairing, variant):
    """MLA rows: latent bit-exact, rope slice rotated; 3 layers, 2,000 tokens of
    16..128-token chunks behind a 32-token leading chunk (carve-out)."""
    base = W.deepseek_v3_mla(context_tokens=2000, num_layers=3)
    m = W.Model("mla-small", "mla", 3, 1, 576, 64, 512, pairing, 1e4, 16)
    wl = W.Workload(f"mla-small-{pairing}", m, base.chunk_lens, base.requests, 0, 32)
    st = Stitched(wl, pool_device="cpu").run()
    try:
        segs, tables, rec = oracle_side(wl, st.nb)
        want_k, _ = oracle.stitch_paged(bits(st.k_pool), None, segs, tables, st.nb, st.bs,
                                        theta_of(m), pairing_of(m), 512, 64)
        got = f64(st.k_cache)
        written = ~np.isnan(want_k[..., 0])
        # latent: bit-exact copy
        gb = bits(st.k_cache)
        wb = np.where(np.isnan(want_k), 0, want_k)
        assert np.array_equal(got[..., :512][written], wb[..., :512][written])
        assert_k_close(got[..., 512:], want_k[..., 512:], "k_r")
        assert np.all(gb[~written] == 0xFFFF)
        assert st.ridx.cpu().numpy()[:st.n_rec].tolist() == rec[0] == list(range(32))
    finally:
        st.close()


def _sample_rows(st, segs, tables, n, seed, shift=None):
    """n random (request, layer, position) picks plus every segment's first and
    last token in random layers: returns index arrays and deltas."""
    rng = np.random.default_rng(seed)
    L = st.m.num_layers
    picks = []
    flat = [(r, j) for r in range(len(segs)) for j in range(len(segs[r])) if segs[r][j].length > 0]
    for (r, j) in flat:
        s = segs[r][j]
        for t in {0, s.length - 1}:
            picks.append((r, j, t, int(rng.integers(L))))
    for _ in range(n):
        r, j = flat[int(rng.integers(len(flat)))]
        picks.append((r, j, int(rng.integers(segs[r][j].length)), int(rng.integers(L))))
    l_idx, blk, row, src, delta = [], [], [], [], []
    for (r, j, t, l) in picks:
        s = segs[r][j]
        p = s.dst_pos + t
        l_idx.append(l)
        blk.append(tables[r][p // st.bs])
        row.append(p % st.bs)
        src.append(s.src_tok + t)
        delta.append(s.delta + (shift[r][j] if shift is not None else 0))
    as_t = lambda a: torch.as_tensor(np.asarray(a, dtype=np.int64), device=DEV)
    return as_t(l_idx), as_t(blk), as_t(row), as_t(src), delta


def _check_sampled(st, segs, tables, n, seed, shift=None):
    l_idx, blk, row, src, delta = _sample_rows(st, segs, tables, n, seed, shift)
    got = f64(st.k_cache[l_idx, blk, row])
    pool = bits(st.k_pool[l_idx, src])
    theta, pairing = theta_of(st.m), pairing_of(st.m)
    off, rd = st.m.rope_offset, st.m.rope_dim
    want = np.stack([oracle.expected_row(pool[i], delta[i], theta, pairing, off, rd) for i in range(len(delta))])
    if shift is None:
        assert_k_close(got, want, "K sampled")
    else:
        # two roundings to bf16 (stitch, then shift), each at most 2^-8 relative per
        # element, so per RoPE pair |err| <= 2 * 2^-8 |pair| (+ fp32 noise)
        ok, worst = _pairs_close(got[..., off:off + rd], want[..., off:off + rd], pairing, 2.0 ** -7 * 1.01)
        assert ok, worst
    if st.m.kind == "mla":
        assert np.array_equal(bits(st.k_cache[l_idx, blk, row])[..., :512], pool[..., :512])
    else:
        assert np.array_equal(bits(st.v_cache[l_idx, blk, row]), bits(st.v_pool[l_idx, src]))
    return len(delta)


def test_mla_full_size_sampled():
    """DeepSeek-V3 MLA shapes at full size: 61 layers x 65,536 tokens."""
    wl = W.deepseek_v3_mla()
    st = Stitched(wl).run()
    try:
        segs, tables, rec = oracle_side(wl, st.nb)
        np.testing.assert_array_equal(st.tables[0][:len(tables[0])], tables[0])
        _check_sampled(st, segs, tables, 4000, 1)
        assert st.ridx.cpu().numpy()[:st.n_rec].tolist() == rec[0]
        assert st.indptr.cpu().tolist() == [0, 32]
    finally:
        st.close()
        del st
        torch.cuda.empty_cache()


def test_qwen3_8b_batch_full_size_sampled():
    """Qwen3-8B shapes at full size: 8 requests x 32,768 tokens, 36 layers."""
    wl = W.qwen3_8b_batch()
    st = Stitched(wl).run()
    try:
        segs, tables, rec = oracle_side(wl, st.nb)
        for r in range(len(tables)):
            np.testing.assert_array_equal(st.tables[r][:len(tables[r])], tables[r])
        _check_sampled(st, segs, tables, 6000, 2)
        indptr, idx = oracle.recompute_csr(rec)
        assert st.indptr.cpu().tolist() == indptr.tolist()
        assert st.ridx.cpu().numpy()[:st.n_rec].tolist() == idx.tolist()
    finally:
        st.close()
        del st
        torch.cuda.empty_cache()


# ----------------------------------------------------------------- in place

@pytest.mark.parametrize("kind,pairing", [("gqa", "neox"), ("gqa", "interleaved"), ("mla", "interleaved"),
                                          ("mla", "neox")])
def test_inplace_parity(kind, pairing, variant):
    """Random cache contents; listed token ranges rotate by their delta
    (|delta| up to 2^17, negative included), every other row is untouched."""
    L, bs = 3, 16
    if kind == "gqa":
        m = W.Model("ip", "gqa", L, 4, 128, 128, 0, pairing, 5e5, bs, W.LLAMA3_SCALING)
    else:
        m = W.Model("ip", "mla", L, 1, 576, 64, 512, pairing, 1e4, bs)
    nb = 40
    ctx = pic.create_from_spec(pic.model_spec_from(m), nb)
    try:
        shape = (L, nb, bs) + tuple(m.row_shape)
        cache = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
        W.fill_random_bf16(cache, 3, "inplace")
        before = bits(cache)
        tables = [list(range(39, 19, -1)), list(range(0, 20))]   # 2 requests x 20 blocks
        segs = [(0, 0, 5, 131072), (0, 5, 40, -131000), (0, 100, 1, 7), (1, 17, 300, 99999),
                (1, 317, 2, 0), (0, 45, 20, -1)]
        ws = torch.empty(pic.pic_rerotate_workspace_bytes(ctx, segs), dtype=torch.uint8, device=DEV)
        bt = torch.tensor(tables, dtype=torch.int32, device=DEV)
        pic.pic_rerotate_inplace(ctx, cache, bt, segs, ws)
        assert pic.pic_query_device_status(ctx, ws) == 0
        want = oracle.rerotate_inplace(before, tables, segs, bs, theta_of(m), pairing_of(m),
                                       m.rope_offset, m.rope_dim)
        got = f64(cache)
        assert_k_close(got, want, "in place")
        listed = np.zeros((nb, bs), bool)
        for (r, s, n, d) in segs:
            for p in range(s, s + n):
                if d != 0:
                    listed[tables[r][p // bs], p % bs] = True
        assert np.array_equal(bits(cache)[:, ~listed], before[:, ~listed])
        if kind == "mla":
            assert np.array_equal(bits(cache)[..., :512], before[..., :512])
    finally:
        pic.pic_destroy(ctx)


def test_serving_stress_full_size_stitch_then_shift():
    """Serving stress at full size (64 x 16,384 tokens, Zipf reuse, 256-chunk
    pool, Llama-3.1-8B shapes): stitch, check a sample; then shift every chunk
    in place to a new position up to 128k and check the sampled rows against
    the oracle's in-place rotation of their own pre-shift bits, per element,
    and against R(delta + delta') of the pool row (EPIC guide: angles add)."""
    wl = W.serving_stress()
    st = Stitched(wl).run()
    try:
        segs, tables, rec = oracle_side(wl, st.nb)
        for r in range(len(tables)):
            np.testing.assert_array_equal(st.tables[r][:len(tables[r])], tables[r])
        _check_sampled(st, segs, tables, 6000, 3)
        indptr, idx = oracle.recompute_csr(rec)
        assert st.ridx.cpu().numpy()[:st.n_rec].tolist() == idx.tolist()
        # in-place mode: chunk j of request r moves to new_pos[r][j]
        shift = [[wl.new_pos[r][j] - s.dst_pos for j, s in enumerate(segs[r])] for r in range(len(segs))]
        shift_segs = [(r, s.dst_pos, s.length, shift[r][j]) for r in range(len(segs))
                      for j, s in enumerate(segs[r])]
        # the rows the checks sample, with their bits before the shift
        l_idx, blk, row, _, d_stitch = _sample_rows(st, segs, tables, 6000, 4)
        _, _, _, _, d_total = _sample_rows(st, segs, tables, 6000, 4, shift=shift)
        pre = bits(st.k_cache[l_idx, blk, row])
        ws = torch.empty(pic.pic_rerotate_workspace_bytes(st.ctx, shift_segs), dtype=torch.uint8, device=DEV)
        pic.pic_rerotate_inplace(st.ctx, st.k_cache, st.d_bt, shift_segs, ws)
        assert pic.pic_query_device_status(st.ctx, ws) == 0
        assert max(abs(d) for _, _, _, d in shift_segs) > 100000
        # (1) the contract: the oracle's in-place rotation R(delta') of the
        # cache's own bits before the shift, per element
        theta, pairing = theta_of(st.m), pairing_of(st.m)
        want = np.stack([oracle.expected_row(pre[i], d_total[i] - d_stitch[i], theta, pairing, 0, 128)
                         for i in range(len(pre))])
        assert_k_close(f64(st.k_cache[l_idx, blk, row]), want, "in place, from the cache's own bits")
        # (2) the composition R(delta') R(delta) = R(delta + delta') of the pool row
        _check_sampled(st, segs, tables, 6000, 4, shift=shift)
    finally:
        st.close()
        del st
        torch.cuda.empty_cache()


def test_stitch_then_shift_composes_small(variant):
    """stitch(delta) then shift(delta') equals R(delta + delta') of the pool
    to two bf16 roundings (2 * 2^-8 per RoPE pair), on every row."""
    wl = _custom_workload("compose", "gqa", 2, 2, 128, "neox", 16, [50, 30, 70], [[(2, 70), (0, 50), (1, 30)]])
    st = Stitched(wl, pool_device="cpu").run()
    try:
        segs, tables, _ = oracle_side(wl, st.nb)
        shift = [[1000, -77777, 131072]]
        shift_segs = [(0, s.dst_pos, s.length, shift[0][j]) for j, s in enumerate(segs[0])]
        ws = torch.empty(pic.pic_rerotate_workspace_bytes(st.ctx, shift_segs), dtype=torch.uint8, device=DEV)
        pic.pic_rerotate_inplace(st.ctx, st.k_cache, st.d_bt, shift_segs, ws)
        assert pic.pic_query_device_status(st.ctx, ws) == 0
        composed = [[oracle.Segment(s.chunk, s.src_tok, s.length, s.dst_pos, s.delta + shift[0][j])
                     for j, s in enumerate(segs[0])]]
        want_k, _ = oracle.stitch_paged(bits(st.k_pool), bits(st.v_pool), composed, tables, st.nb, 16,
                                        theta_of(wl.model), oracle.NEOX_HALF, 0, 128)
        got = f64(st.k_cache)
        m = ~np.isnan(want_k[..., 0])
        ok, worst = _pairs_close(got[m], want_k[m], oracle.NEOX_HALF, 2.0 ** -7 * 1.01)
        assert ok, worst
    finally:
        st.close()
