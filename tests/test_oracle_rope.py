"""Pins of the oracle's RoPE frequencies and rotation against facts that do
not come from the oracle itself: closed forms, textbook formulations (complex
multiplication; GPT-NeoX rotate-half), the group law, norms and relative
position.  A dropped term, a flipped sign, a swapped pair index or a wrong
frequency index each fails at least one of these."""

import itertools
import math

import numpy as np
import pytest

import oracle
import workloads as W
from oracle import INTERLEAVED, NEOX_HALF


# ---------------------------------------------------------------- frequencies

def test_inv_freq_closed_form_power_of_two_base():
    # b = 2^d makes theta_i = 2^(-2i) exactly (EPIC guide: theta_i = b^(-2i/d)).
    for d in (4, 8, 16, 64, 128):
        th = oracle.rope_inv_freq(d, 2.0 ** d)
        assert th.shape == (d // 2,)
        np.testing.assert_array_equal(th, [2.0 ** (-2 * i) for i in range(d // 2)])


def test_inv_freq_first_is_one_and_geometric():
    for d, b in ((128, 1e4), (128, 5e5), (64, 1e4), (128, 1e6)):
        th = oracle.rope_inv_freq(d, b)
        assert th[0] == 1.0
        # last frequency b^-(d-2)/d and constant ratio b^(-2/d)
        assert math.isclose(th[-1], b ** (-(d - 2) / d), rel_tol=1e-14)
        r = th[1:] / th[:-1]
        np.testing.assert_allclose(r, b ** (-2.0 / d), rtol=1e-13)


def test_inv_freq_listing_values_base_1e4():
    # The EPIC listing's EPICConfig: head_dim 128, rope_base 10000; theta_32 = 1e4^(-1/2) = 0.01.
    th = oracle.rope_inv_freq(128, 10000.0)
    assert math.isclose(th[32], 0.01, rel_tol=1e-14)
    assert math.isclose(th[16], 0.1, rel_tol=1e-14)


def test_llama3_invariants():
    """Parity unpinned rule (not on the pages): only its regime invariants are tested."""
    th = oracle.rope_inv_freq(128, 5e5)
    sc = oracle.llama3_inv_freq(th, 8.0, 1.0, 4.0, 8192)
    wl = 2 * math.pi / th
    hi = wl < 8192 / 4
    lo = wl > 8192 / 1
    np.testing.assert_array_equal(sc[hi], th[hi])
    np.testing.assert_allclose(sc[lo], th[lo] / 8.0, rtol=1e-15)
    mid = ~hi & ~lo
    assert mid.any()
    assert np.all(sc[mid] <= th[mid]) and np.all(sc[mid] >= th[mid] / 8.0)
    # monotone non-increasing frequencies after scaling
    assert np.all(np.diff(sc) <= 0)


def test_llama3_continuous_at_both_regime_boundaries():
    """The blend meets the kept frequencies at wavelength orig/high and the
    divided ones at orig/low; between them theta'/theta is affine in theta
    (s is linear in orig/lambda).  A swapped low/high, a sign slip in s or a
    blend weighted the wrong way round breaks one of these."""
    orig, factor, low, high = 8192, 8.0, 1.0, 4.0
    for lam, left, right in ((orig / high, 1.0, 1.0), (orig / low, 1.0 / factor, 1.0 / factor)):
        for eps in (1e-6, 1e-9):
            th = np.array([2 * math.pi / (lam * (1 - eps)), 2 * math.pi / (lam * (1 + eps))])
            sc = oracle.llama3_inv_freq(th, factor, low, high, orig) / th
            assert abs(sc[0] - left) < 10 * eps and abs(sc[1] - right) < 10 * eps
    th = 2 * math.pi / np.linspace(orig / high * 1.01, orig / low * 0.99, 9)
    ratio = oracle.llama3_inv_freq(th, factor, low, high, orig) / th
    slope = np.diff(ratio) / np.diff(th)
    np.testing.assert_allclose(slope, slope[0], rtol=1e-9)
    assert slope[0] > 0  # higher frequency, less division


# Hand-derived values of the Llama-3.1 rule with orig 8192, low 1, high 4,
# factor 8.  At wavelength lambda, s = (8192 / lambda - 1) / 3 and
# theta' / theta = (1 - s) / 8 + s.  Choosing 8192 / lambda = 1.75, 2.5 and
# 3.25 puts s at exactly 1/4, 1/2 and 3/4:
#   s = 1/4: 3/32 + 8/32 = 11/32 = 0.34375
#   s = 1/2: 1/16 + 8/16 =  9/16 = 0.5625
#   s = 3/4: 1/32 + 24/32 = 25/32 = 0.78125
# lambda = 8192 gives s = 0 (1/8) and lambda = 2048 gives s = 1 (1), so the
# blend meets both outer regimes; lambda = 2000 (< 8192 / 4) keeps theta and
# lambda = 9000 (> 8192 / 1) divides it by 8.  A swapped low/high keeps
# theta at 8192/3.25 ~ 2521 (ratio 1, not 25/32); a blend weighted the wrong
# way round gives 25/32 at s = 1/4.
LLAMA3_HAND = [(2000.0, 1.0), (2048.0, 1.0), (8192 / 3.25, 0.78125), (8192 / 2.5, 0.5625),
               (8192 / 1.75, 0.34375), (8192.0, 0.125), (9000.0, 0.125)]


def test_llama3_hand_derived_ratios():
    lam = np.array([w for w, _ in LLAMA3_HAND])
    want = np.array([r for _, r in LLAMA3_HAND])
    th = 2 * math.pi / lam
    got = oracle.llama3_inv_freq(th, 8.0, 1.0, 4.0, 8192) / th
    np.testing.assert_allclose(got, want, rtol=1e-12)


def test_llama3_factor_one_is_the_identity():
    """With factor 1 every regime gives theta back: theta/1, or
    (1 - s) theta + s theta."""
    th = oracle.rope_inv_freq(128, 5e5)
    np.testing.assert_allclose(oracle.llama3_inv_freq(th, 1.0, 1.0, 4.0, 8192), th, rtol=1e-15)


def test_llama3_regimes_of_the_llama31_table():
    """Llama-3.1-8B's table (base 5e5, d = 128): lambda_i = 2 pi 5e5^(i/64).
    By hand, ln 5e5 = 13.1224, so lambda_28 = 2 pi e^5.741 = 1956 < 2048,
    lambda_29 = 2 pi e^5.946 = 2402 > 2048, lambda_34 = 2 pi e^6.971 = 6695
    < 8192 and lambda_35 = 2 pi e^7.176 = 8219 > 8192: frequencies 0-28 are
    kept, 35-63 divided by 8, and 29-34 blended, strictly between."""
    th = oracle.rope_inv_freq(128, 5e5)
    r = oracle.model_inv_freq(128, 5e5, W.LLAMA3_SCALING) / th
    np.testing.assert_array_equal(r[:29], 1.0)
    np.testing.assert_allclose(r[35:], 0.125, rtol=1e-15)
    assert np.all((r[29:35] > 0.125) & (r[29:35] < 1.0))


def test_model_table_end_entries_closed_forms():
    """theta_0 = b^0 = 1 in every table; Llama-3.1's highest frequency has a
    wavelength of 2 pi < 8192/4 and is kept, its lowest (wavelength about
    3.3e5 > 8192) is divided by the factor 8."""
    plain = oracle.model_inv_freq(128, 5e5)
    sc = oracle.model_inv_freq(128, 5e5, W.LLAMA3_SCALING)
    assert plain[0] == 1.0 and sc[0] == 1.0
    assert math.isclose(plain[-1], 5e5 ** (-126 / 128), rel_tol=1e-14)
    assert math.isclose(sc[-1], 5e5 ** (-126 / 128) / 8.0, rel_tol=1e-14)
    assert len(sc) == 64


@pytest.mark.parametrize("pairing", [NEOX_HALF, INTERLEAVED])
def test_expected_row_identity_and_quarter_turn(pairing):
    """An MLA-shaped row (576 dims, rope slice at 512..575): delta 0 returns
    the bf16 values exactly; with every frequency pi/2 a shift of 1 maps each
    rope pair (x, y) to (-y, x) and leaves the latent alone."""
    rng = np.random.default_rng(3)
    bits = (rng.standard_normal(576).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x = oracle.bf16_bits_to_f64(bits)
    th = np.full(32, math.pi / 2)
    np.testing.assert_array_equal(oracle.expected_row(bits, 0, th, pairing, 512, 64), x)
    got = oracle.expected_row(bits, 1, th, pairing, 512, 64)
    np.testing.assert_array_equal(got[:512], x[:512])
    a, b = oracle.rope_pairs(64, pairing)
    np.testing.assert_allclose(got[512 + a], -x[512 + b], atol=1e-15)
    np.testing.assert_allclose(got[512 + b], x[512 + a], atol=1e-15)


# ------------------------------------------------------------ rotation basics

@pytest.mark.parametrize("pairing", [NEOX_HALF, INTERLEAVED])
def test_delta_zero_is_identity(pairing):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 128))
    th = oracle.rope_inv_freq(128, 1e4)
    np.testing.assert_array_equal(oracle.rotate(x, 0, th, pairing), x)


def test_quarter_turn_closed_forms_interleaved():
    # theta = (pi/2, pi, 3pi/2, 2pi): delta = 1 turns the planes by 90, 180, 270, 360 degrees.
    th = np.array([0.5, 1.0, 1.5, 2.0]) * math.pi
    x = np.array([1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0, 8.0])
    y = oracle.rotate(x, 1, th, INTERLEAVED)
    expect = np.array([-2.0, 1.0, -3.0, -4.0, 6.0, -5.0, 7.0, 8.0])
    np.testing.assert_allclose(y, expect, atol=1e-14)


def test_quarter_turn_closed_forms_neox():
    th = np.array([0.5, 1.0, 1.5, 2.0]) * math.pi
    x = np.array([1.0, 3.0, 5.0, 7.0, 2.0, 4.0, 6.0, 8.0])  # pairs (1,2) (3,4) (5,6) (7,8)
    y = oracle.rotate(x, 1, th, NEOX_HALF)
    expect = np.array([-2.0, -3.0, 6.0, 7.0, 1.0, -4.0, -5.0, 8.0])
    np.testing.assert_allclose(y, expect, atol=1e-14)


def test_negative_delta_is_transpose():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 64))
    th = oracle.rope_inv_freq(64, 1e4)
    for p in (NEOX_HALF, INTERLEAVED):
        y = oracle.rotate(oracle.rotate(x, 777, th, p), -777, th, p)
        np.testing.assert_allclose(y, x, atol=1e-12)


def _rope_complex(raw, m, theta, pairing):
    """Textbook RoPE as complex multiplication: plane i is the complex number
    z_i, rotated to z_i * exp(i m theta_i)."""
    d = raw.shape[-1]
    h = d // 2
    if pairing == INTERLEAVED:
        z = raw[..., 0::2] + 1j * raw[..., 1::2]
    else:
        z = raw[..., :h] + 1j * raw[..., h:]
    z = z * np.exp(1j * np.float64(m) * theta)
    out = np.empty_like(raw)
    if pairing == INTERLEAVED:
        out[..., 0::2] = z.real
        out[..., 1::2] = z.imag
    else:
        out[..., :h] = z.real
        out[..., h:] = z.imag
    return out


def _rope_rotate_half(raw, m, theta):
    """GPT-NeoX / Llama forward RoPE: x*cos + rotate_half(x)*sin, where
    rotate_half(x) = [-x2, x1] and cos/sin repeat the d/2 angles twice."""
    ang = np.concatenate([m * theta, m * theta])
    h = raw.shape[-1] // 2
    rot = np.concatenate([-raw[..., h:], raw[..., :h]], axis=-1)
    return raw * np.cos(ang) + rot * np.sin(ang)


def _rope_listing_restated(raw, m, theta):
    """The EPIC listing's rotation, restated: even coordinates get
    e*cos - o*sin, odd coordinates e*sin + o*cos, angle m*theta_i."""
    e = raw[..., 0::2]
    o = raw[..., 1::2]
    out = np.empty_like(raw)
    out[..., 0::2] = e * np.cos(m * theta) - o * np.sin(m * theta)
    out[..., 1::2] = e * np.sin(m * theta) + o * np.cos(m * theta)
    return out


def _angle_tol(n, dp, raw):
    """fp64 forms m*theta with |m*theta| <= |m| (theta_0 = 1): the two sides'
    angles differ by a few ulp(|n| + |dp|), which moves a value by at most
    that many radians times the pair norm."""
    ulps = 8.0 * 2.0 ** -52 * (abs(n) + abs(dp) + 1.0)
    return 1e-14 + ulps * 2.0 * np.max(np.abs(raw))


@pytest.mark.parametrize("d,base", [(128, 1e4), (128, 5e5), (64, 1e4), (256, 1e6)])
def test_shift_of_cached_key_equals_key_at_shifted_position(d, base):
    """EPIC guide, In-Place Shift Transformation: R_dp (R_n k_raw) = R_{n+dp} k_raw,
    checked against two independent forward-RoPE formulations."""
    rng = np.random.default_rng(3)
    th = oracle.rope_inv_freq(d, base)
    raw = rng.standard_normal(d)
    for n, dp in [(0, 1), (0, 128), (5, 8320), (1000, -999), (17, 131072), (0, -131072), (3, 2 ** 24 - 1)]:
        for pairing in (NEOX_HALF, INTERLEAVED):
            cached = _rope_complex(raw, n, th, pairing)
            got = oracle.rotate(cached, dp, th, pairing)
            want = _rope_complex(raw, n + dp, th, pairing)
            np.testing.assert_allclose(got, want, atol=_angle_tol(n, dp, raw))
        want_rh = _rope_rotate_half(raw, n + dp, th)
        got_rh = oracle.rotate(_rope_rotate_half(raw, n, th), dp, th, NEOX_HALF)
        np.testing.assert_allclose(got_rh, want_rh, atol=_angle_tol(n, dp, raw))


def test_interleaved_matches_listing_rotation_on_raw_keys():
    """The EPIC listing rotates token n by angle (dp + n) theta_i; on raw
    (unrotated) keys that is forward RoPE at position dp + n.  The oracle
    must agree with it there."""
    rng = np.random.default_rng(4)
    th = oracle.rope_inv_freq(128, 10000.0)
    raw = rng.standard_normal((6, 128))
    dp = 4096
    for n in range(6):
        np.testing.assert_allclose(oracle.rotate(raw[n], dp + n, th, INTERLEAVED),
                                   _rope_listing_restated(raw[n], dp + n, th), atol=1e-12)


def test_composition_brute_force_tiny():
    """R(a) R(b) = R(a + b) for every a, b in [-64, 64] (EPIC guide: angles add)."""
    rng = np.random.default_rng(5)
    th = oracle.rope_inv_freq(8, 10.0)
    x = rng.standard_normal(8)
    for pairing in (NEOX_HALF, INTERLEAVED):
        for a, b in itertools.product(range(-64, 65), range(-64, 65)):
            y = oracle.rotate(oracle.rotate(x, a, th, pairing), b, th, pairing)
            np.testing.assert_allclose(y, oracle.rotate(x, a + b, th, pairing), atol=1e-12)


def test_pair_norms_preserved():
    """R_m is orthogonal and block-diagonal: each plane keeps its length."""
    rng = np.random.default_rng(6)
    th = oracle.rope_inv_freq(128, 1e4)
    x = rng.standard_normal((4, 128))
    for pairing in (NEOX_HALF, INTERLEAVED):
        a, b = oracle.rope_pairs(128, pairing)
        y = oracle.rotate(x, 12345, th, pairing)
        np.testing.assert_allclose(np.hypot(y[:, a], y[:, b]), np.hypot(x[:, a], x[:, b]), rtol=1e-13)


def test_pairs_partition_the_dims():
    for d in (8, 64, 128):
        for pairing in (NEOX_HALF, INTERLEAVED):
            a, b = oracle.rope_pairs(d, pairing)
            assert sorted(np.concatenate([a, b]).tolist()) == list(range(d))


def test_dot_product_depends_only_on_relative_position():
    """q.k after RoPE at (m, n) equals the same at (m + s, n + s)."""
    rng = np.random.default_rng(7)
    th = oracle.rope_inv_freq(128, 5e5)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for pairing in (NEOX_HALF, INTERLEAVED):
        for m, n, s in [(10, 3, 100), (0, 500, 70000), (4096, 128, -4000)]:
            d1 = oracle.rotate(q, m, th, pairing) @ oracle.rotate(k, n, th, pairing)
            d2 = oracle.rotate(q, m + s, th, pairing) @ oracle.rotate(k, n + s, th, pairing)
            assert math.isclose(d1, d2, rel_tol=1e-9, abs_tol=1e-9)


def test_mla_rows_rotate_only_rope_slice():
    """Irminsul: the 512-d latent is reused verbatim, only the 64-d k_r turns."""
    rng = np.random.default_rng(8)
    th = oracle.rope_inv_freq(64, 1e4)
    rows = rng.standard_normal((3, 576))
    out = oracle.rotate_rows(rows, 9999, th, INTERLEAVED, 512, 64)
    np.testing.assert_array_equal(out[:, :512], rows[:, :512])
    np.testing.assert_allclose(out[:, 512:], oracle.rotate(rows[:, 512:], 9999, th, INTERLEAVED))
    assert not np.allclose(out[:, 512:], rows[:, 512:])


def test_bf16_decode_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x7F7F, 0x0001], dtype=np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    assert vals[0] == 1.0 and vals[1] == -1.0 and vals[3] == 0.0
    assert vals[2] == 3.140625
    assert math.copysign(1.0, vals[4]) == -1.0
    assert vals[5] == float.fromhex("0x1.fep127")
    assert vals[6] == float.fromhex("0x1p-133")
