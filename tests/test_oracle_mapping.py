"""Pins of the oracle's virtual block mapping: the block ids printed on the
EPIC runtime figure, forward RoPE at the mapped positions, and the
exclusivity rules that keep in-place rotations race-free."""

import numpy as np
import pytest

import oracle
from oracle import BlockChunk, BlockPool, Chunk, NEOX_HALF
from conftest import load_golden


def _figure_chunks():
    g = load_golden("epic_virtual_block_mapping.json")
    ch = g["chunks"]
    mk = lambda d: tuple(d["blocks"]) if "blocks" in d else tuple(range(d["blocks_range"][0], d["blocks_range"][1] + 1))
    chunks = {name: BlockChunk(mk(d), d["num_tokens"], d["base_pos"]) for name, d in ch.items()}
    return g, chunks


def test_figure_block_mapping_matches_epic_runtime_figure():
    g, chunks = _figure_chunks()
    bs = g["block_size"]
    assert len(chunks["DocA"].blocks) == 47 and len(chunks["DocB"].blocks) == 71
    pool = BlockPool(1024)
    for c in chunks.values():               # the chunks' blocks are taken
        for b in c.blocks:
            pool.free[b] = False
    total = sum(c.num_tokens for c in chunks.values()) + g["query_tokens"]
    assert total == g["expected_total_tokens"]
    segs, table, fresh, _ = oracle.map_request(chunks, g["order"], bs, pool, "req", total_tokens=total)
    assert [s.mode for s in segs] == ["alias"] * 3
    assert [s.dst_pos for s in segs] == g["expected_dst_pos"]
    assert [s.delta for s in segs] == g["expected_delta"]
    want = [102] + list(range(310, 381)) + list(range(204, 251))
    assert table[:len(want)] == want            # "Reuses Physical Blocks 102, 310..380, 204..250"
    assert fresh == [0, 1] and table[len(want):] == [0, 1]   # the 20-token query gets fresh blocks


def _rope(raw, m, theta):
    h = raw.shape[-1] // 2
    z = (raw[..., :h] + 1j * raw[..., h:]) * np.exp(1j * np.float64(m) * theta)
    return np.concatenate([z.real, z.imag], axis=-1)


def _to_bf16_bits(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def test_mapped_and_copied_keys_equal_forward_rope_at_new_positions():
    """Block chunks hold keys rotated to their current position; after the
    request, every key at position p equals the raw key rotated to p, values
    are bit copies, and mapped values never moved."""
    rng = np.random.default_rng(21)
    L, H, D, bs, nb = 2, 1, 16, 4, 24
    theta = oracle.rope_inv_freq(D, 1e4)
    raw = {}
    chunks = {
        "A": BlockChunk((5, 9), 8, cur_pos=40),        # mapped (aligned, whole, unique)
        "B": BlockChunk((11, 12), 6, cur_pos=0),       # lands at 8 + 3 = 11: not aligned -> copied
        "P": Chunk(0, 3, 0),                           # a pool chunk
    }
    pool = BlockPool(nb)
    for name in ("A", "B"):
        for b in chunks[name].blocks:
            pool.free[b] = False
    kc = np.zeros((L, nb, bs, H, D))
    vc = rng.integers(0, 1 << 16, size=(L, nb, bs, H, D), dtype=np.uint16)
    for name in ("A", "B"):
        c = chunks[name]
        raw[name] = rng.standard_normal((L, c.num_tokens, H, D))
        for t in range(c.num_tokens):
            kc[:, c.blocks[t // bs], t % bs] = _rope(raw[name][:, t], c.cur_pos + t, theta)
    raw["P"] = rng.standard_normal((L, 3, H, D))
    k_pool = np.stack([_rope(raw["P"][:, t], t, theta) for t in range(3)], axis=1)
    v_pool = rng.integers(0, 1 << 16, size=(L, 3, H, D), dtype=np.uint16)
    kb, kpb = _to_bf16_bits(kc), _to_bf16_bits(k_pool)
    segs, table, fresh, undo = oracle.map_request(chunks, ["A", "P", "B"], bs, pool, "r1")
    assert [s.mode for s in segs] == ["alias", "copy", "copy"]
    assert [s.src_kind for s in segs] == ["", "pool", "cache"]
    assert table[0:2] == [5, 9]
    k_out, v_out = oracle.apply_mapped(kb, vc, kpb, v_pool, segs, table, bs, theta, NEOX_HALF, 0, D)
    for s in segs:
        for t in range(s.length):
            p = s.dst_pos + t
            slot, row = table[p // bs], p % bs
            want = _rope(raw[s.chunk][:, t], p, theta)
            a, b = oracle.rope_pairs(D, NEOX_HALF)
            err = np.hypot(k_out[:, slot, row][..., a] - want[..., a], k_out[:, slot, row][..., b] - want[..., b])
            assert np.all(err <= 2.0 ** -8 * np.hypot(want[..., a], want[..., b]) + 1e-12)
            if s.mode == "alias":
                assert np.array_equal(v_out[:, slot, row], vc[:, slot, row])     # values never move
            elif s.src_kind == "cache":
                c = chunks[s.chunk]
                assert np.array_equal(v_out[:, slot, row], vc[:, c.blocks[t // bs], t % bs])
            else:
                assert np.array_equal(v_out[:, slot, row], v_pool[:, t])
    assert chunks["A"].cur_pos == 0 and chunks["A"].mapped_by == "r1"
    assert chunks["B"].cur_pos == 0 and chunks["B"].refs == 1


def test_exclusivity_refs_and_undo():
    bs = 4
    chunks = {"X": BlockChunk((3, 4), 8, cur_pos=100), "Y": Chunk(0, 5, 0)}
    pool = BlockPool(16)
    for b in (3, 4):
        pool.free[b] = False
    # A maps X; B may not use X while A lives
    sa, ta, fa, ua = oracle.map_request(chunks, ["X", "Y"], bs, pool, "A")
    assert sa[0].mode == "alias" and sa[0].delta == -100 and chunks["X"].cur_pos == 0
    with pytest.raises(oracle.BusyError):
        oracle.map_request(chunks, ["Y", "X"], bs, pool, "B")
    # A freed without its rotation applied: X goes back to position 100
    oracle.release_request(chunks, sa, fa, ua, pool, applied=False)
    assert chunks["X"].cur_pos == 100 and chunks["X"].mapped_by is None and chunks["X"].refs == 0
    # A again, applied: X stays at 0
    sa, ta, fa, ua = oracle.map_request(chunks, ["X"], bs, pool, "A")
    oracle.release_request(chunks, sa, fa, ua, pool, applied=True)
    assert chunks["X"].cur_pos == 0
    # a live copy of X forbids mapping it (its rows may still be read)
    sc, tc, fc, uc = oracle.map_request(chunks, ["Y", "X"], bs, pool, "C")     # position 5: copy
    assert sc[1].mode == "copy" and chunks["X"].refs == 1
    sd, td, fd, ud = oracle.map_request(chunks, ["X"], bs, pool, "D")
    assert sd[0].mode == "copy"
    # two occurrences in one request: both copied
    oracle.release_request(chunks, sc, fc, uc, pool, applied=True)
    oracle.release_request(chunks, sd, fd, ud, pool, applied=True)
    se, te, fe, ue = oracle.map_request(chunks, ["X", "X"], bs, pool, "E")
    assert [s.mode for s in se] == ["copy", "copy"]
    # aliasing off: copied
    oracle.release_request(chunks, se, fe, ue, pool, applied=True)
    sf, tf, ff, uf = oracle.map_request(chunks, ["X"], bs, pool, "F", alias=False)
    assert sf[0].mode == "copy"
