"""Pins of the oracle's cached-key rerotation and int8 requantisation."""
import math

import numpy as np
import pytest

from oracle.sinkkv_oracle import (RopeSpec, dequantize_int8_rows, dynamic_factor, quantize_int8_rows,
                                  rerotate, rerotate_int8, rope_inv_freq, rope_rotate)

# The cached-key rerotation configuration: r=64 of d_h=128, YaRN L0=262144, factor 1 -> 2.
SPEC_A = RopeSpec(128, 64, 5e5, True, 1.0, 262144)
SPEC_B = SPEC_A.with_factor(2.0)


def _keys(n, seed=4):
    rng = np.random.default_rng(seed)
    return rng.uniform(-1, 1, size=(n, 4, 128)), rng.integers(0, 524288, size=n)


def test_rerotated_equals_rotated_from_raw():
    """Turning keys stored at factor A equals rotating the raw key at factor B
    ("Attention Sink 与 Streaming KV Cache": rerotation vs recompute from raw K)."""
    raw, pos = _keys(64)
    a = rope_rotate(raw, pos, SPEC_A.omega(), SPEC_A.mscale(), 64)
    b = rope_rotate(raw, pos, SPEC_B.omega(), SPEC_B.mscale(), 64)
    # positions reach 524287, so angles reach ~5e5 rad: float64 angle error ~1e-10
    np.testing.assert_allclose(rerotate(a, pos, SPEC_A, SPEC_B), b, rtol=0, atol=1e-9)
    small = np.arange(64) % 50
    a = rope_rotate(raw, small, SPEC_A.omega(), SPEC_A.mscale(), 64)
    b = rope_rotate(raw, small, SPEC_B.omega(), SPEC_B.mscale(), 64)
    np.testing.assert_allclose(rerotate(a, small, SPEC_A, SPEC_B), b, rtol=0, atol=1e-13)
    assert np.array_equal(rerotate(a, small, SPEC_A, SPEC_B)[..., 64:], raw[..., 64:])


def test_round_trip_and_chain():
    raw, pos = _keys(32, seed=7)
    a = rope_rotate(raw, pos, SPEC_A.omega(), 1.0, 64)
    back = rerotate(rerotate(a, pos, SPEC_A, SPEC_B), pos, SPEC_B, SPEC_A)
    np.testing.assert_allclose(back, a, atol=1e-9)
    # the seven-switch chain of "#2961" (1 -> 1.125 -> ... -> 2) equals one 1 -> 2 turn
    chain = [1.0, 1.125, 1.25, 1.5, 1.625, 1.75, 1.875, 2.0]
    k = a
    for fa, fb in zip(chain[:-1], chain[1:]):
        k = rerotate(k, pos, SPEC_A.with_factor(fa), SPEC_A.with_factor(fb))
    np.testing.assert_allclose(k, rerotate(a, pos, SPEC_A, SPEC_B), atol=1e-9)


def test_local_shift_by_minus_one():
    """Local-position implementations shift recent keys from [3,4,5] to [2,3,4]
    with a rotation by -1 (GPT-J pairing, d=8, base 1e4, as in the page-4
    experiment); skipping it changes the scores by well over 1e-3."""
    rng = np.random.default_rng(229)
    d = 8
    om = rope_inv_freq(d, 1e4)
    raw = rng.standard_normal((3, 1, d))
    old = rope_rotate(raw, [3, 4, 5], om, 1.0, d, neox=False)
    shifted = rope_rotate(old, [-1, -1, -1], om, 1.0, d, neox=False)
    recomputed = rope_rotate(raw, [2, 3, 4], om, 1.0, d, neox=False)
    np.testing.assert_allclose(shifted, recomputed, atol=1e-12)
    query = rope_rotate(rng.standard_normal((1, 1, d)), [5], om, 1.0, d, neox=False)[0, 0]
    wrong = old[:, 0] @ query / math.sqrt(d)
    right = shifted[:, 0] @ query / math.sqrt(d)
    assert np.abs(right - wrong).max() > 1e-3


def test_int8_quantisation_rules():
    s = 2.0 ** -3
    # ties round half to even: 2.5 -> 2, 3.5 -> 4, -2.5 -> -2; the max maps to 127
    row = np.array([[127 * s, 2.5 * s, 3.5 * s, -2.5 * s, 0.0, -127 * s]])
    codes, scale = quantize_int8_rows(row)
    assert scale[0] == np.float32(s)
    assert codes[0].tolist() == [127, 2, 4, -2, 0, -127]
    z, zs = quantize_int8_rows(np.zeros((1, 8)))
    assert zs[0] == 1.0 and not z.any()
    x = np.random.default_rng(1).uniform(-3, 3, size=(200, 128))
    c, sc = quantize_int8_rows(x)
    assert c.min() >= -127 and c.max() <= 127
    assert np.all(np.abs(c).max(axis=1) == 127)
    err = np.abs(dequantize_int8_rows(c, sc) - x)
    assert np.all(err <= sc[:, None] * (0.5 + 1e-5))


def test_int8_rerotation_error_within_page_bounds():
    """Turned-from-A against written-at-B, both measured against the float64 key
    at B ("#2961", rope_dynamic_parity): RMS ratio <= 1.6x, worst <= 2 steps."""
    raw, pos = _keys(4000, seed=9)
    exact_b = rope_rotate(raw, pos, SPEC_B.omega(), SPEC_B.mscale(), 64)
    written_b_codes, written_b_scale = quantize_int8_rows(exact_b)
    a = rope_rotate(raw, pos, SPEC_A.omega(), SPEC_A.mscale(), 64)
    ca, sa = quantize_int8_rows(a)
    cb, sb, _ = rerotate_int8(ca, sa, pos, SPEC_A, SPEC_B)
    turned = dequantize_int8_rows(cb, sb)
    written = dequantize_int8_rows(written_b_codes, written_b_scale)
    rms_t = np.sqrt(np.mean((turned - exact_b) ** 2))
    rms_w = np.sqrt(np.mean((written - exact_b) ** 2))
    assert 1.0 < rms_t / rms_w <= 1.6
    worst_steps = np.max(np.abs(turned - exact_b) / written_b_scale[..., None])
    assert worst_steps <= 2.0


def test_bf16_like_rerotation_error_within_page_bounds():
    """The same yardstick for 16-bit keys: a turn re-rounds once more, so its
    RMS error is about sqrt(2) that of a key written directly at B."""
    raw, pos = _keys(4000, seed=10)

    def round_bf16(x):
        b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
        b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
        return b.astype(np.uint32).view(np.float32).astype(np.float64)

    exact_b = rope_rotate(raw, pos, SPEC_B.omega(), SPEC_B.mscale(), 64)
    a = round_bf16(rope_rotate(raw, pos, SPEC_A.omega(), SPEC_A.mscale(), 64))
    turned = round_bf16(rerotate(a, pos, SPEC_A, SPEC_B))
    written = round_bf16(exact_b)
    rms_t = np.sqrt(np.mean((turned - exact_b) ** 2))
    rms_w = np.sqrt(np.mean((written - exact_b) ** 2))
    assert 1.0 < rms_t / rms_w <= 1.6


def test_dynamic_factor_policy():
    from tests.conftest import golden_path
    with open(golden_path("dynamic_factor_values.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for total, l0, step, cap, want in rows:
        assert dynamic_factor(int(total), int(l0), float(step), float(cap)) == float(want)
    # the switch chain of the page's growing dialog is a subset of the policy's values
    seen = {dynamic_factor(p, 262144, 0.125, 2.0) for p in range(262144, 524289, 4096)}
    assert {1.125, 1.25, 1.5, 1.625, 1.75, 1.875, 2.0} <= seen


def _local_ring(S, W, T, seed, neox=True, r=64, D=128):
    """A ring whose keys are rotated at their local positions: sinks at 0..S-1, the
    recent keys at S.. in chronological order (the local-position scheme of page 4),
    plus the raw keys by absolute position."""
    from oracle.sinkkv_oracle import RingCache
    rng = np.random.default_rng(seed)
    raw = rng.standard_normal((T, 2, D))
    v = rng.standard_normal((T, 2, D))
    ring = RingCache(S, W)
    ring.append([(raw[t], v[t]) for t in range(T)])
    om = rope_inv_freq(r, 1e4)
    local = {}
    for i, s in enumerate(ring.chronological_slots()):
        P = ring.slot_pos[s]
        local[s] = i
        k, vv = ring.slots[s]
        ring.slots[s] = (rope_rotate(k[None], [i], om, 1.0, r, neox)[0], vv)
    return ring, raw, v, om, local


@pytest.mark.parametrize("neox", [True, False])
def test_shift_recent_equals_recompute_at_local_minus_one(neox):
    """Page 4's C=6, S=2 cache after 10 tokens: recent keys (absolute 6..9) sit at
    local positions 2..5; shifting them by -1 equals rotating their raw keys at local
    1..4 (1e-12); sink keys and every value stay bit for bit."""
    from oracle.sinkkv_oracle import shift_recent_keys
    ring, raw, v, om, local = _local_ring(2, 4, 10, 7, neox)
    assert [ring.slot_pos[s] for s in ring.chronological_slots()] == [0, 1, 6, 7, 8, 9]
    before = {s: (ring.slots[s][0].copy(), ring.slots[s][1]) for s in range(ring.C)}
    shift_recent_keys(ring, -1, om, 64, neox)
    for s in range(ring.C):
        k, vv = ring.slots[s]
        assert vv is before[s][1]
        P = ring.slot_pos[s]
        if s < ring.S:
            np.testing.assert_array_equal(k, before[s][0])
        else:
            want = rope_rotate(raw[P][None], [local[s] - 1], om, 1.0, 64, neox)[0]
            np.testing.assert_allclose(k, want, atol=1e-12)


def test_shift_recent_there_and_back_and_partial_ring():
    """+3 then -3 is the identity; a ring that has not wrapped turns only its
    occupied slots (count < W)."""
    from oracle.sinkkv_oracle import shift_recent_keys
    ring, raw, v, om, local = _local_ring(3, 8, 7, 8)
    assert ring.count == 4
    before = [None if x is None else x[0].copy() for x in ring.slots]
    shift_recent_keys(ring, 3, om, 64)
    for s in range(ring.S, ring.S + ring.count):
        assert np.abs(ring.slots[s][0] - before[s]).max() > 1e-3
    for s in range(ring.S + ring.count, ring.C):
        assert ring.slots[s] is None
    shift_recent_keys(ring, -3, om, 64)
    for s in range(ring.S + ring.count):
        np.testing.assert_allclose(ring.slots[s][0], before[s], atol=1e-12)
