"""Pins of the oracle's composer, block allocator and recompute list against
the numbers the pages print and against brute force on tiny requests."""

import itertools

import numpy as np
import pytest

import oracle
from oracle import BlockPool, Chunk
from conftest import load_golden


def test_composer_matches_epic_composition_figure():
    g = load_golden("epic_composition_figure.json")
    chunks = [Chunk(0, c["num_tokens"], c["base_pos"]) for c in g["chunks"]]
    segs = oracle.compose(chunks, g["order"], start_pos=g["start_pos"])
    assert [s.dst_pos for s in segs] == g["expected_dst_pos"]
    assert [s.delta for s in segs] == g["expected_delta"]


def test_composer_and_sinks_match_epic_listing():
    g = load_golden("epic_listing_sinks.json")
    chunks, off = [], 0
    for n in g["doc_tokens"]:
        chunks.append(Chunk(off, n, 0))
        off += n
    segs = oracle.compose(chunks, range(len(chunks)))
    assert [s.dst_pos for s in segs] == g["expected_dst_pos"]
    assert [s.delta for s in segs] == g["expected_delta"]
    assert oracle.recompute_positions(segs, g["sink_tokens"], 0) == g["expected_recompute"]


def test_explicit_offsets_match_epic_client_request():
    g = load_golden("epic_client_request.json")
    n = g["chunk_tokens"]
    chunks = [Chunk(0, n, 0), Chunk(n, n, 0)]
    segs = oracle.compose(chunks, [0, 1], dst_pos=g["offsets"])
    assert [s.delta for s in segs] == g["expected_delta"]
    assert oracle.recompute_positions(segs, g["sink_tokens"], 0) == g["expected_recompute"]


def test_irminsul_first_chunk_carve_out():
    g = load_golden("irminsul_carve_out.json")
    for case in g["cases"]:
        chunks, off = [], 0
        for n in case["chunk_tokens"]:
            chunks.append(Chunk(off, n, 0))
            off += n
        segs = oracle.compose(chunks, range(len(chunks)))
        got = oracle.recompute_positions(segs, case["k_nonleading"], case["k_leading"])
        assert got == case["expected_recompute"]
    row = g["mla_row"]
    total = row["latent_dims"] + row["rope_dims"]
    assert abs(row["latent_dims"] / total - row["latent_share_approx"]) < 0.005
    assert abs(row["rope_dims"] / total - row["rope_share_approx"]) < 0.005


def test_base_pos_gives_signed_delta():
    # Irminsul: delta = p_target - p_source; a chunk computed at 500 placed at 100 turns back.
    chunks = [Chunk(0, 64, 0), Chunk(64, 32, 500)]
    segs = oracle.compose(chunks, [0, 1], start_pos=36)
    assert [(s.dst_pos, s.delta) for s in segs] == [(36, 36), (100, -400)]


def test_composer_rejects_overlap_and_overtake():
    chunks = [Chunk(0, 10), Chunk(10, 10)]
    with pytest.raises(ValueError):
        oracle.compose(chunks, [0, 1], dst_pos=[0, 5])
    with pytest.raises(ValueError):
        oracle.compose(chunks, [0], take=[11])


def test_take_truncates_and_zero_length():
    chunks = [Chunk(0, 10), Chunk(10, 7)]
    segs = oracle.compose(chunks, [1, 0, 1], take=[3, 0, 7])
    assert [(s.src_tok, s.length, s.dst_pos) for s in segs] == [(10, 3, 0), (0, 0, 3), (10, 7, 3)]
    # a zero-length segment contributes no recompute tokens
    assert oracle.recompute_positions(segs, 4, 2) == [0, 1, 3, 4, 5, 6]


def test_recompute_clamps_to_segment_length():
    chunks = [Chunk(0, 2), Chunk(2, 3), Chunk(5, 9)]
    segs = oracle.compose(chunks, [0, 1, 2], start_pos=0)
    assert oracle.recompute_positions(segs, 4, 0) == [2, 3, 4, 5, 6, 7, 8]


def test_recompute_brute_force_count_and_order():
    for lens in itertools.product([0, 1, 3, 4, 5, 16], repeat=3):
        chunks, off = [], 0
        for n in lens:
            chunks.append(Chunk(off, n))
            off += n
        for start in (0, 5):
            segs = oracle.compose(chunks, range(3), start_pos=start)
            for k, kl in ((4, 0), (0, 32), (2, 3)):
                got = oracle.recompute_positions(segs, k, kl)
                want = []
                for s in segs:
                    kk = kl if s.dst_pos == 0 else k
                    want += [p for p in range(s.dst_pos, s.dst_pos + s.length)
                             if p - s.dst_pos < kk]
                assert got == want
                assert got == sorted(got) and len(set(got)) == len(got)


def test_block_pool_lowest_first_brute_force():
    """Every allocate/free sequence over a tiny pool: blocks are distinct, the
    count is ceil(T / block_size), and each request takes the lowest free ids."""
    bs = 4
    for totals in itertools.product([0, 1, 4, 5, 9], repeat=3):
        for free_mask in range(8):
            pool = BlockPool(12)
            used = set()
            tables = []
            for t in totals:
                n = oracle.blocks_needed(t, bs)
                assert n == (t + bs - 1) // bs
                free_before = sorted(set(range(12)) - used)
                ids = pool.allocate(n)
                assert ids == free_before[:n]
                used |= set(ids)
                tables.append(ids)
            for i, ids in enumerate(tables):
                if free_mask >> i & 1:
                    pool.release(ids)
                    used -= set(ids)
            again = pool.allocate(2)
            assert again == sorted(set(range(12)) - used)[:2]


def test_block_pool_exhaustion_and_double_free():
    pool = BlockPool(3)
    ids = pool.allocate(3)
    with pytest.raises(MemoryError):
        pool.allocate(1)
    pool.release(ids[:1])
    with pytest.raises(ValueError):
        pool.release(ids[:1])


def test_recompute_csr_layout():
    indptr, idx = oracle.recompute_csr([[1, 2], [], [7]])
    assert indptr.tolist() == [0, 2, 2, 3]
    assert idx.tolist() == [1, 2, 7]
