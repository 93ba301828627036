"""End-to-end pins of the oracle's stitch and in-place shift.

Pool keys are made the way the pages describe cached chunks: raw keys rotated
to their local positions n = 0 .. len-1 (forward RoPE written here as complex
multiplication, independent of the oracle).  After stitching, the key at
absolute position p must be the raw key rotated to p (EPIC guide, In-Place
Shift Transformation), values must be the pool's bits (values untouched), and
nothing outside the request's slots may change."""

import numpy as np

import oracle
from oracle import BlockPool, Chunk, INTERLEAVED, NEOX_HALF


def _rope_complex(raw, m, theta, pairing):
    d = raw.shape[-1]
    h = d // 2
    if pairing == INTERLEAVED:
        z = raw[..., 0::2] + 1j * raw[..., 1::2]
    else:
        z = raw[..., :h] + 1j * raw[..., h:]
    z = z * np.exp(1j * np.float64(m) * theta)
    out = np.empty_like(raw)
    if pairing == INTERLEAVED:
        out[..., 0::2], out[..., 1::2] = z.real, z.imag
    else:
        out[..., :h], out[..., h:] = z.real, z.imag
    return out


def _to_bf16_bits(x):
    """Round float64 -> float32 (nearest) -> bfloat16 (nearest-even) bits."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _pair_err_ok(got, want, pairing, rel):
    a, b = oracle.rope_pairs(got.shape[-1], pairing)
    err = np.hypot(got[..., a] - want[..., a], got[..., b] - want[..., b])
    norm = np.hypot(want[..., a], want[..., b])
    return np.all(err <= rel * norm + 1e-12)


def _build(lens, order, start_pos, bs, num_blocks, base_pos=None):
    chunks, off = [], 0
    for i, n in enumerate(lens):
        chunks.append(Chunk(off, n, 0 if base_pos is None else base_pos[i]))
        off += n
    segs = oracle.compose(chunks, order, start_pos=start_pos)
    total = segs[-1].dst_pos + segs[-1].length
    pool = BlockPool(num_blocks)
    bt = pool.allocate(oracle.blocks_needed(total, bs))
    return chunks, segs, bt, off


def test_gqa_stitch_equals_forward_rope_at_target():
    rng = np.random.default_rng(11)
    L, H, D, bs = 2, 2, 16, 4
    theta = oracle.rope_inv_freq(D, 1e4)
    lens = [5, 9, 3]
    for pairing in (NEOX_HALF, INTERLEAVED):
        chunks, segs, bt, P = _build(lens, [2, 0, 1], 0, bs, 10)
        raw = rng.standard_normal((L, P, H, D))
        k_pool = np.empty((L, P, H, D))
        for c in chunks:
            for n in range(c.num_tokens):
                k_pool[:, c.pool_offset + n] = _rope_complex(raw[:, c.pool_offset + n], n, theta, pairing)
        kb = _to_bf16_bits(k_pool)
        vb = rng.integers(0, 1 << 16, size=(L, P, H, D), dtype=np.uint16)
        k_out, v_out = oracle.stitch_paged(kb, vb, [segs], [bt], 10, bs, theta, pairing, 0, D)
        written = set()
        for s in segs:
            for t in range(s.length):
                p = s.dst_pos + t
                slot, row = bt[p // bs], p % bs
                written.add((slot, row))
                want = _rope_complex(raw[:, s.src_tok + t], p, theta, pairing)
                assert _pair_err_ok(k_out[:, slot, row], want, pairing, 2.0 ** -8)
                np.testing.assert_array_equal(v_out[:, slot, row], vb[:, s.src_tok + t])
        for slot in range(10):
            for row in range(bs):
                if (slot, row) not in written:
                    assert np.all(np.isnan(k_out[:, slot, row]))
                    assert np.all(v_out[:, slot, row] == oracle.BF16_SENTINEL)


def test_mla_stitch_rotates_rope_copies_latent():
    rng = np.random.default_rng(12)
    L, bs = 2, 4
    theta = oracle.rope_inv_freq(64, 1e4)
    lens = [6, 7]
    chunks, segs, bt, P = _build(lens, [1, 0], 3, bs, 8)
    raw = rng.standard_normal((L, P, 64))
    rows = rng.standard_normal((L, P, 576))
    for c in chunks:
        for n in range(c.num_tokens):
            rows[:, c.pool_offset + n, 512:] = _rope_complex(raw[:, c.pool_offset + n], n, theta, INTERLEAVED)
    kb = _to_bf16_bits(rows)
    k_out, v_out = oracle.stitch_paged(kb, None, [segs], [bt], 8, bs, theta, INTERLEAVED, 512, 64)
    assert v_out is None
    for s in segs:
        for t in range(s.length):
            p = s.dst_pos + t
            slot, row = bt[p // bs], p % bs
            np.testing.assert_array_equal(k_out[:, slot, row, :512],
                                          oracle.bf16_bits_to_f64(kb[:, s.src_tok + t, :512]))
            want = _rope_complex(raw[:, s.src_tok + t], p, theta, INTERLEAVED)
            assert _pair_err_ok(k_out[:, slot, row, 512:], want, INTERLEAVED, 2.0 ** -8)
    # positions before start_pos (inline tokens) are not written
    for p in range(3):
        assert np.all(np.isnan(k_out[:, bt[p // bs], p % bs]))


def test_chunk_cached_at_nonzero_base_pos():
    """A chunk computed at base position 40 and placed at 7 is rotated by -33."""
    rng = np.random.default_rng(13)
    D, bs = 8, 4
    theta = oracle.rope_inv_freq(D, 100.0)
    chunks, segs, bt, P = _build([4, 5], [0, 1], 3, bs, 4, base_pos=[0, 40])
    raw = rng.standard_normal((1, P, 1, D))
    k_pool = np.empty_like(raw)
    for c in chunks:
        for n in range(c.num_tokens):
            k_pool[:, c.pool_offset + n] = _rope_complex(raw[:, c.pool_offset + n], c.base_pos + n, theta, NEOX_HALF)
    kb = _to_bf16_bits(k_pool)
    k_out, _ = oracle.stitch_paged(kb, None, [segs], [bt], 4, bs, theta, NEOX_HALF, 0, D)
    assert segs[1].delta == 7 - 40
    for s in segs:
        for t in range(s.length):
            p = s.dst_pos + t
            want = _rope_complex(raw[:, s.src_tok + t], p, theta, NEOX_HALF)
            assert _pair_err_ok(k_out[:, bt[p // bs], p % bs], want, NEOX_HALF, 2.0 ** -8)


def test_inplace_shift_moves_keys_and_nothing_else():
    rng = np.random.default_rng(14)
    L, nb, bs, H, D = 2, 6, 4, 2, 16
    theta = oracle.rope_inv_freq(D, 1e4)
    raw = rng.standard_normal((L, nb, bs, H, D))
    # cache rows hold keys at their logical positions p of request 0 (table [4, 1, 5])
    bt = [[4, 1, 5]]
    cache = np.zeros_like(raw)
    for p in range(12):
        cache[:, bt[0][p // bs], p % bs] = _rope_complex(raw[:, bt[0][p // bs], p % bs], p, theta, NEOX_HALF)
    bits = _to_bf16_bits(cache)
    before = oracle.bf16_bits_to_f64(bits)
    segs = [(0, 2, 7, 1000), (0, 10, 1, -10)]
    out = oracle.rerotate_inplace(bits, bt, segs, bs, theta, NEOX_HALF, 0, D)
    moved = set()
    for (req, start, n, d) in segs:
        for t in range(n):
            p = start + t
            slot, row = bt[req][p // bs], p % bs
            moved.add((slot, row))
            want = _rope_complex(raw[:, slot, row], p + d, theta, NEOX_HALF)
            assert _pair_err_ok(out[:, slot, row], want, NEOX_HALF, 2.0 ** -8)
    for slot in range(nb):
        for row in range(bs):
            if (slot, row) not in moved:
                np.testing.assert_array_equal(out[:, slot, row], before[:, slot, row])
