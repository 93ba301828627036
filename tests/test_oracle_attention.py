"""Pins of the oracle's decode attention and LegoLink sink bias."""

import math

import numpy as np

import oracle
from oracle import Chunk, NEOX_HALF


def test_uniform_scores_average_values():
    rng = np.random.default_rng(31)
    v = rng.standard_normal((7, 2, 16))
    k = np.zeros((7, 2, 16))                         # every score 0
    out, lse = oracle.attention_decode(rng.standard_normal((4, 16)), k, v, 0.25)
    np.testing.assert_allclose(out[0], v[:, 0].mean(axis=0), atol=1e-14)
    np.testing.assert_allclose(out[3], v[:, 1].mean(axis=0), atol=1e-14)   # head 3 reads KV head 1
    np.testing.assert_allclose(lse, math.log(7), atol=1e-14)


def test_dominant_score_selects_its_value():
    rng = np.random.default_rng(32)
    v = rng.standard_normal((5, 1, 8))
    k = np.zeros((5, 1, 8))
    k[3, 0, 0] = 1000.0
    q = np.zeros((1, 8))
    q[0, 0] = 1.0
    out, _ = oracle.attention_decode(q, k, v, 1.0)
    np.testing.assert_allclose(out[0], v[3, 0], atol=1e-12)


def test_token_order_does_not_matter():
    rng = np.random.default_rng(33)
    q, k, v = rng.standard_normal((8, 32)), rng.standard_normal((20, 2, 32)), rng.standard_normal((20, 2, 32))
    perm = rng.permutation(20)
    a, la = oracle.attention_decode(q, k, v, 0.2)
    b, lb = oracle.attention_decode(q, k[perm], v[perm], 0.2)
    np.testing.assert_allclose(a, b, atol=1e-13)
    np.testing.assert_allclose(la, lb, atol=1e-13)


def test_shifting_query_and_keys_together_is_invisible():
    """RoPE attention depends only on relative positions: query at m, keys at
    n_t versus query at m + s, keys at n_t + s (EPIC Guide: R_n^T R_m = R_{m-n})."""
    rng = np.random.default_rng(34)
    D, T = 64, 12
    theta = oracle.rope_inv_freq(D, 1e4)
    raw_q, raw_k, v = rng.standard_normal((2, D)), rng.standard_normal((T, 1, D)), rng.standard_normal((T, 1, D))
    pos = np.arange(T) * 3 + 5
    def run(shift):
        qq = oracle.rotate(raw_q, 100 + shift, theta, NEOX_HALF)
        kk = np.stack([oracle.rotate(raw_k[t], pos[t] + shift, theta, NEOX_HALF) for t in range(T)])
        return oracle.attention_decode(qq, kk, v, 1 / 8)
    a, la = run(0)
    b, lb = run(70000)
    np.testing.assert_allclose(a, b, atol=1e-9)
    np.testing.assert_allclose(la, lb, atol=1e-9)


def test_sink_bias_follows_the_listing_boundary_loop():
    chunks = [Chunk(0, 10), Chunk(10, 3), Chunk(13, 20)]
    segs = oracle.compose(chunks, [0, 1, 2])
    b = oracle.sink_bias(segs, 40, 4, -15.0)
    want = np.zeros(40)
    want[10:13] = -15.0        # chunk 1 is only 3 tokens long
    want[13:17] = -15.0        # chunk 2: its first 4 tokens
    np.testing.assert_array_equal(b, want)       # chunk 0 (global token 0) untouched


def test_mla_absorbed_attention_equals_per_head_attention():
    """Irminsul 2.1 (MLA decomposition): a head's key is [W_UK c | k_r] and its
    value W_UV c.  With the query absorbed, q_abs = [W_UK^T q_nope | q_rope],
    attention over the shared latent rows [c | k_r] gives the same scores, and
    W_UV applied to its latent output gives the head's output -- the form the
    MLA decode attention computes (values = the latent)."""
    rng = np.random.default_rng(35)
    T, dc, dr, dn, dv = 9, 16, 4, 6, 5
    w_uk, w_uv = rng.standard_normal((dn, dc)), rng.standard_normal((dv, dc))
    c, k_r = rng.standard_normal((T, dc)), rng.standard_normal((T, dr))
    q_nope, q_rope = rng.standard_normal(dn), rng.standard_normal(dr)
    keys = np.concatenate([c @ w_uk.T, k_r], axis=1)[:, None, :]
    vals = (c @ w_uv.T)[:, None, :]
    want, want_lse = oracle.attention_decode(np.concatenate([q_nope, q_rope])[None], keys, vals, 0.3)
    rows = np.concatenate([c, k_r], axis=1)[:, None, :]
    q_abs = np.concatenate([w_uk.T @ q_nope, q_rope])[None]
    lat, lse = oracle.attention_decode(q_abs, rows, c[:, None, :], 0.3)
    np.testing.assert_allclose(lat @ w_uv.T, want, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse, atol=1e-12)
