"""Pins of the oracle's paged-cache functions: block counts printed on the pages, the
static-sink metadata rule, and equality with the contiguous caches' attention."""
import numpy as np
import pytest

from oracle.sinkkv_oracle import (GlobalCache, RingCache, attend, blocks_for_tokens, decode_attention,
                                  first_window_token, paged_decode_attention, paged_logical_rows,
                                  prefill_attention, prepend_static_sinks, visible_positions, window_blocks)


def test_page_block_counts(golden):
    g = golden("paged_block_counts.txt")
    assert window_blocks(4096, 16) == int(g["window_blocks_w4096_bs16"])
    assert blocks_for_tokens(131072, 16) == int(g["full_blocks_131072_bs16"])


def test_window_block_bound_holds_for_every_alignment():
    """Brute force: the W newest tokens of any length touch at most window_blocks(W, bs)
    blocks, and some length reaches the bound."""
    for bs in (1, 4, 16):
        for W in range(1, 70):
            worst = 0
            for L in range(1, 200):
                keys = range(max(0, L - W), L)
                worst = max(worst, len({k // bs for k in keys}))
            assert worst <= window_blocks(W, bs)
            assert worst >= window_blocks(W, bs) - 1


def test_first_window_token_is_the_oldest_visible_recent_key():
    for W in (1, 3, 8):
        for P in range(W, 60):
            vis = visible_positions(P, W, 0)          # S = 0: a pure window of W
            assert first_window_token(P, W) == vis[0]


def test_prepend_static_sinks_rule():
    table = np.array([[7, 3, 9], [2, 5, 1], [4, 4, 4]])
    tab, lens = prepend_static_sinks(table, [0, 5, 17], [11], 16)
    assert lens.tolist() == [0, 21, 33]                # a zero length stays zero
    assert tab.tolist() == [[11, 7, 3, 9], [11, 2, 5, 1], [11, 4, 4, 4]]


def _pool(n_blocks, Hkv, bs, D, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n_blocks, Hkv, bs, D)), rng.standard_normal((n_blocks, Hkv, bs, D))


def test_logical_rows_follow_the_block_table():
    """Scatter a contiguous sequence into a permuted pool, then gather it back."""
    rng = np.random.default_rng(1)
    bs, Hkv, D, L = 4, 2, 8, 37
    rows_k = rng.standard_normal((L, Hkv, D))
    rows_v = rng.standard_normal((L, Hkv, D))
    nb = blocks_for_tokens(L, bs)
    perm = rng.permutation(20)[:nb]
    kp = np.zeros((20, Hkv, bs, D))
    vp = np.zeros((20, Hkv, bs, D))
    for i in range(L):
        kp[perm[i // bs], :, i % bs] = rows_k[i]
        vp[perm[i // bs], :, i % bs] = rows_v[i]
    k, v = paged_logical_rows(kp, vp, perm, L, bs)
    np.testing.assert_array_equal(k, rows_k)
    np.testing.assert_array_equal(v, rows_v)


@pytest.mark.parametrize("S,W,L", [(4, 20, 63), (4, 20, 10), (0, 16, 50), (2, 5, 6)])
def test_paged_decode_equals_ring_decode(S, W, L):
    """Request sinks + window over a paged cache equal the contiguous ring cache with
    the same keys; freed blocks (outside the visible set) may hold anything."""
    bs, Hkv, Hq, D = 4, 2, 4, 8
    rng = np.random.default_rng(2)
    kp, vp = _pool(40, Hkv, bs, D, 3)
    table = rng.permutation(40)[:blocks_for_tokens(L, bs)]
    q = rng.standard_normal((Hq, D))
    want_k, want_v = paged_logical_rows(kp, vp, table, L, bs)
    ring = RingCache(S, W)
    ring.append([(want_k[i], want_v[i]) for i in range(L)])
    got = paged_decode_attention(q, kp, vp, table, L, bs, S, W)
    np.testing.assert_allclose(got, decode_attention(ring, q), atol=1e-12)
    # blocks holding no visible key are freed: point them at garbage
    vis = set(visible_positions(L - 1, S + W, S))
    garbage = 39
    kp[garbage] = 1e6
    freed = np.array([b if any((j * bs + o) in vis for o in range(bs)) else garbage
                      for j, b in enumerate(table)])
    np.testing.assert_allclose(paged_decode_attention(q, kp, vp, freed, L, bs, S, W), got, atol=1e-12)


def test_paged_decode_full_attention_and_static_sinks():
    """window None = every key (the global cache); static sink blocks in front of the
    table with sinks = sink_len equal the dense sink mask on the concatenated keys."""
    bs, Hkv, Hq, D = 4, 2, 4, 8
    rng = np.random.default_rng(4)
    kp, vp = _pool(30, Hkv, bs, D, 5)
    q = rng.standard_normal((Hq, D))
    table = rng.permutation(30)[:7]
    L = 26
    k, v = paged_logical_rows(kp, vp, table, L, bs)
    g = GlobalCache(64)
    g.append([(k[i], v[i]) for i in range(L)])
    np.testing.assert_allclose(paged_decode_attention(q, kp, vp, table, L, bs, 0, None),
                               decode_attention(g, q), atol=1e-12)
    # two static sink blocks (8 tokens) prepended, window of 6 over the request's keys
    sink_blocks = [28, 29]
    tab, lens = prepend_static_sinks(table[None, :6], [19], sink_blocks, 8)
    Lt = int(lens[0])
    got = paged_decode_attention(q, kp, vp, tab[0], Lt, bs, 8, 6)
    kk, vv = paged_logical_rows(kp, vp, tab[0], Lt, bs)
    qs = np.zeros((Lt, Hq, D))
    qs[-1] = q
    dense = prefill_attention(qs, kk, vv, 0, 8, 6, rows=[Lt - 1])[0]
    np.testing.assert_allclose(got, dense, atol=1e-12)
    # a request with no tokens attends to nothing
    assert not paged_decode_attention(q, kp, vp, tab[0], 0, bs, 8, 6).any()
