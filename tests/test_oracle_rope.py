"""Pins of the oracle's RoPE / YaRN arithmetic against the pages and against
mathematics that does not go through the oracle's own formulas."""
import math

import numpy as np
import pytest

from oracle.sinkkv_oracle import (RopeSpec, kv_bytes_per_token, rope_inv_freq, rope_rotate,
                                  yarn_correction_dim, yarn_correction_range, yarn_inv_freq,
                                  yarn_linear_ramp, yarn_mscale)


def _floats(s):
    return [float(x) for x in s.split(",")]


def test_worked_number_pair16(golden):
    g = golden("rope_yarn_worked_values.txt")
    om = rope_inv_freq(128, 1e4)
    assert om[16] == pytest.approx(float(g["omega16_b1e4_r128"]), rel=1e-14)
    assert 2 * math.pi / om[16] == pytest.approx(float(g["wavelength16_b1e4_r128"]), abs=0.05)


@pytest.mark.parametrize("m,n,key", [(5, 3, "score_q5_k3"), (105, 103, "score_q105_k103")])
def test_worked_score_is_cos02(golden, m, n, key):
    g = golden("rope_yarn_worked_values.txt")
    D = r = 128
    om = rope_inv_freq(r, 1e4)
    q = np.zeros((1, 1, D))
    k = np.zeros((1, 1, D))
    q[0, 0, 16] = 1.0   # NeoX pair 16 = (x_16, x_80); (1, 0) before rotation
    k[0, 0, 16] = 1.0
    qr = rope_rotate(q, [m], om, 1.0, r, neox=True)
    kr = rope_rotate(k, [n], om, 1.0, r, neox=True)
    score = float(qr[0, 0] @ kr[0, 0])
    assert score == pytest.approx(float(g[key]), abs=5e-8)
    # the vectors themselves moved: they are no longer (1, 0)
    assert abs(qr[0, 0, 16] - 1.0) > 0.1


@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("r,D", [(64, 64), (64, 128), (128, 128)])
def test_rotation_is_complex_multiplication(neox, r, D):
    """Each pair (x1, x2) read as x1 + i x2 is multiplied by mu * exp(i P omega)."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((7, 3, D))
    pos = rng.integers(0, 600000, size=7)
    spec = RopeSpec(D, r, 5e5, neox, yarn_factor=2.0, yarn_orig_ctx=262144)
    om, mu = spec.omega(), spec.mscale()
    y = rope_rotate(x, pos, om, mu, r, neox)
    if neox:
        z = x[..., : r // 2] + 1j * x[..., r // 2: r]
        w = y[..., : r // 2] + 1j * y[..., r // 2: r]
    else:
        z = x[..., 0:r:2] + 1j * x[..., 1:r:2]
        w = y[..., 0:r:2] + 1j * y[..., 1:r:2]
    expect = z * mu * np.exp(1j * (pos[:, None, None] * om[None, None, :]))
    np.testing.assert_allclose(w, expect, rtol=0, atol=1e-9)
    # the tail passes through bit for bit
    assert np.array_equal(y[..., r:], x[..., r:])


@pytest.mark.parametrize("neox", [True, False])
def test_relative_position_invariance(neox):
    """q at m against k at n depends on m - n only (p1: 5 vs 3 equals 105 vs 103)."""
    rng = np.random.default_rng(3)
    D, r = 128, 128
    om = rope_inv_freq(r, 1e4)
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, 1, D))
    base = None
    for m in [5, 105, 4101, 77777]:
        n = m - 2
        s = float(rope_rotate(q, [m], om, 1.0, r, neox)[0, 0] @ rope_rotate(k, [n], om, 1.0, r, neox)[0, 0])
        if base is None:
            base = s
        assert s == pytest.approx(base, abs=1e-9)
    # and it does depend on the distance
    s_far = float(rope_rotate(q, [5], om, 1.0, r, neox)[0, 0] @ rope_rotate(k, [0], om, 1.0, r, neox)[0, 0])
    assert abs(s_far - base) > 1e-3


def test_rotation_scales_norm_by_mscale_and_composes():
    rng = np.random.default_rng(5)
    D, r = 128, 64
    x = rng.standard_normal((4, 2, D))
    pos = [0, 1, 1000, 524287]
    spec = RopeSpec(D, r, 5e5, True, 2.0, 262144)
    y = rope_rotate(x, pos, spec.omega(), spec.mscale(), r, True)
    np.testing.assert_allclose(np.linalg.norm(y[..., :r], axis=-1),
                               spec.mscale() * np.linalg.norm(x[..., :r], axis=-1), rtol=1e-13)
    # R(a) R(b) = R(a + b)
    om = rope_inv_freq(r, 1e4)
    a = rope_rotate(rope_rotate(x, [3, 4, 5, 6], om, 1.0, r), [10, 20, 30, 40], om, 1.0, r)
    b = rope_rotate(x, [13, 24, 35, 46], om, 1.0, r)
    np.testing.assert_allclose(a, b, atol=1e-12)
    # position 0 is the identity
    z = rope_rotate(x, [0, 0, 0, 0], om, 1.0, r)
    np.testing.assert_allclose(z, x, atol=0)


def test_yarn_band_worked_example(golden):
    g = golden("rope_yarn_worked_values.txt")
    assert yarn_correction_dim(32, 128, 1e4, 4096) == pytest.approx(float(g["yarn_d32_r128_b1e4_L4096"]), abs=0.005)
    assert yarn_correction_dim(1, 128, 1e4, 4096) == pytest.approx(float(g["yarn_d1_r128_b1e4_L4096"]), abs=0.005)
    assert list(yarn_correction_range(32, 1, 128, 1e4, 4096)) == _floats(g["yarn_band_r128_b1e4_L4096"])
    assert list(yarn_correction_range(32, 1, 128, 5e5, 4096)) == _floats(g["yarn_band_r128_b5e5_L4096"])
    assert list(yarn_correction_range(32, 1, 128, 5e5, 8192)) == _floats(g["yarn_band_r128_b5e5_L8192"])


def test_yarn_band_rotation_counts(golden):
    """Rotations in L0 of the band's edge pairs: L0 * omega_i / (2 pi)."""
    g = golden("rope_yarn_worked_values.txt")
    om = rope_inv_freq(128, 1e4)
    rot = [4096 * om[i] / (2 * math.pi) for i in (20, 21, 45, 46)]
    for got, want in zip(rot, _floats(g["rotations_pairs_20_21_45_46"])):
        assert got == pytest.approx(want, abs=0.005)
    assert 2 * math.pi / om[21] == pytest.approx(float(g["wavelength21_b1e4_r128"]), abs=0.5)
    assert 2 * math.pi / om[45] == pytest.approx(float(g["wavelength45_b1e4_r128"]), abs=0.5)
    om5 = rope_inv_freq(128, 5e5)
    assert 2 * math.pi / om5[63] == pytest.approx(float(g["wavelength63_b5e5_r128"]), rel=0.005)


def test_yarn_mscale(golden):
    g = golden("rope_yarn_worked_values.txt")
    assert yarn_mscale(8.0) == pytest.approx(float(g["yarn_mscale_s8"]), abs=5e-5)
    assert yarn_mscale(8.0) ** 2 == pytest.approx(float(g["yarn_mscale_sq_s8"]), abs=5e-4)
    assert yarn_mscale(1.0) == 1.0 and yarn_mscale(0.5) == 1.0
    assert yarn_mscale(2.0) == pytest.approx(1.0 + 0.1 * math.log(2.0), rel=1e-15)


def test_yarn_regions_and_degenerate_factor():
    """Pairs up to low keep the plain frequency, pairs from high on are divided by s,
    the band between lies strictly between; s = 1 reduces to plain RoPE."""
    r, theta, L0, s = 128, 1e4, 4096, 8.0
    plain = rope_inv_freq(r, theta)
    y = yarn_inv_freq(r, theta, s, L0)
    low, high = 20, 46
    np.testing.assert_allclose(y[: low + 1], plain[: low + 1], rtol=1e-15)
    np.testing.assert_allclose(y[high:], plain[high:] / s, rtol=1e-15)
    mid = slice(low + 1, high)
    assert np.all(y[mid] < plain[mid]) and np.all(y[mid] > plain[mid] / s)
    np.testing.assert_allclose(yarn_inv_freq(r, theta, 1.0, L0), plain, rtol=1e-15)
    assert np.array_equal(RopeSpec(r, r, theta, yarn_factor=1.0).omega(), plain)


def test_yarn_band_is_linear_in_the_pair_index():
    """Inside the band the page's ramp is linear in i, so omega_i * pos_freq_i =
    1 - ramp_i (1 - 1/s) has zero second differences over pairs low .. high, and at
    the band's midpoint i = 33 of (20, 46) it is exactly halfway between 1 and 1/s
    ("RoPE, scaling, sliding window, attention sinks", "YaRN, precisely")."""
    r, theta, L0, s = 128, 1e4, 4096, 8.0
    y = yarn_inv_freq(r, theta, s, L0)
    pos_freq = theta ** (np.arange(0, r, 2) / r)
    rel = y * pos_freq                     # 1 below the band, 1/s above it
    band = rel[20:47]
    np.testing.assert_allclose(np.diff(band, 2), 0.0, atol=1e-14)
    assert rel[33] == pytest.approx((1.0 + 1.0 / s) / 2.0, rel=1e-14)
    # the step per pair is (1 - 1/s) / (high - low)
    np.testing.assert_allclose(np.diff(band), -(1.0 - 1.0 / s) / 26.0, rtol=1e-12)


def test_yarn_ramp_degenerate_band_is_a_step():
    """low == high: the page's ramp moves high by 0.001 to avoid dividing by zero,
    which makes the ramp a step, 0 up to and including pair low and 1 after it."""
    assert yarn_linear_ramp(5, 5, 10).tolist() == [0.0] * 6 + [1.0] * 4
    assert yarn_linear_ramp(0, 0, 4).tolist() == [0.0, 1.0, 1.0, 1.0]
    # the same branch reached through the whole frequency blend: with L0 = 6 every
    # pair turns less than once in L0 tokens, d(1) < 0 and d(32) < 0, so the band
    # clamps to (0, 0); pair 0 keeps its frequency 1 and every other pair is divided by s
    r, theta, L0, s = 128, 1e4, 6, 4.0
    assert yarn_correction_range(32, 1, r, theta, L0) == (0, 0)
    y = yarn_inv_freq(r, theta, s, L0)
    plain = theta ** (-np.arange(0, r, 2) / r)
    assert y[0] == 1.0
    np.testing.assert_allclose(y[1:], plain[1:] / s, rtol=1e-15)


def test_kv_bytes_context_numbers(golden):
    g = golden("rope_yarn_worked_values.txt")
    assert kv_bytes_per_token(32, 8, 128, 2) == int(g["kv_bytes_per_token_llama3_8b"])
    per_layer_token = kv_bytes_per_token(1, 8, 128, 2)
    hybrid = 8 * 131072 * per_layer_token + 24 * 4096 * per_layer_token
    uniform = 32 * 131072 * per_layer_token
    assert hybrid / 2 ** 30 == float(g["hybrid_gib_128k"])
    assert uniform / 2 ** 30 == float(g["uniform_gib_128k"])


# ---- the cos/sin table -----------------------------------------------------------------

def test_table_worked_number_row(golden):
    """Row P=2, pair 16 (theta 1e4, r 128, omega 0.1) holds (cos 0.2, sin 0.2): the
    page's worked score cos(0.2) for a relative offset of 2."""
    from oracle.sinkkv_oracle import rope_table
    g = golden("rope_yarn_worked_values.txt")
    t = rope_table(RopeSpec(128, 128, 1e4), 3)
    assert t[2, 16, 0] == pytest.approx(float(g["score_q5_k3"]), abs=5e-8)
    assert t[2, 16, 1] == pytest.approx(math.sqrt(1 - float(g["score_q5_k3"]) ** 2), abs=5e-7)
    np.testing.assert_array_equal(t[0, :, 0], np.ones(64))
    np.testing.assert_array_equal(t[0, :, 1], np.zeros(64))


@pytest.mark.parametrize("neox", [True, False])
def test_table_rows_are_the_rotation_of_a_unit_pair(neox):
    """Rotating the unit vector of a pair's first element at P gives the table entry:
    (cos, sin) land in the pair's (first, second) slots."""
    from oracle.sinkkv_oracle import rope_table, rotary_pairs
    spec = RopeSpec(128, 64, 5e5, neox, 2.0, 4096)
    t = rope_table(spec, 40)
    first, second = rotary_pairs(64, neox)
    for j in [0, 7, 31]:
        x = np.zeros((40, 1, 128))
        x[:, 0, first[j]] = 1.0
        y = rope_rotate(x, range(40), spec.omega(), spec.mscale(), 64, neox)
        np.testing.assert_allclose(y[:, 0, first[j]], t[:, j, 0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(y[:, 0, second[j]], t[:, j, 1], rtol=0, atol=1e-15)


def test_table_rows_compose_and_carry_mscale(golden):
    """|row| = mu (0.1 ln s + 1; 1.2079 at s = 8) and row(a) row(b) = mu row(a + b) as
    complex numbers (R_a R_b = R_{a+b})."""
    from oracle.sinkkv_oracle import rope_table
    g = golden("rope_yarn_worked_values.txt")
    t = rope_table(RopeSpec(128, 128, 1e4, True, 8.0, 4096), 300)
    z = t[..., 0] + 1j * t[..., 1]
    np.testing.assert_allclose(np.abs(z), float(g["yarn_mscale_s8"]), atol=5e-5)
    for a, b in [(3, 5), (100, 199), (17, 0)]:
        np.testing.assert_allclose(z[a] * z[b], np.abs(z[0, 0]) * z[a + b], atol=1e-12)
