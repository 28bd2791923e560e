"""Pins of the oracle's chunked prefill over a cached prefix (a prompt chunk that
continues a sequence whose earlier tokens sit in a ring or global cache)."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import (GlobalCache, RingCache, decode_attention, prefill_attention,
                                  prefill_attention_prior, visible_positions)


def _qkv(T, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, Hq, D)), rng.standard_normal((T, Hkv, D)),
            rng.standard_normal((T, Hkv, D)))


def _sdpa_rows(q, k, v, mask):
    """torch float64 SDPA of queries q [Tq, Hq, D] over keys k, v [Tk, Hkv, D] with a
    boolean mask [Tq, Tk] (GQA by repeating kv heads)."""
    n_rep = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(n_rep, 0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(n_rep, 0)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(mask))
    return o.permute(1, 0, 2).numpy()


def _ring_after(k, v, n, S, W, chunks=None):
    c = RingCache(S, W)
    done = 0
    for T in (chunks or [n]):
        c.append([(k[i], v[i]) for i in range(done, done + T)])
        done += T
    assert done == n
    return c


@pytest.mark.parametrize("S,W", [(2, 4), (0, 5), (4, 3), (3, 11)])
def test_chunk_over_ring_equals_rows_of_the_table_mask(S, W):
    """Split a 23-token prompt anywhere: the second chunk, attending over the ring the
    first chunk left, equals the same rows of attention over the whole prompt under the
    page's visible-set table V(P) (capacity S + W), here through torch's SDPA."""
    L, Hq, Hkv, D = 23, 8, 4, 16
    q, k, v = _qkv(L, Hq, Hkv, D, 11)
    mask = np.zeros((L, L), dtype=bool)
    for P in range(L):
        mask[P, visible_positions(P, S + W, S)] = True
    dense = _sdpa_rows(q, k, v, mask)
    for c in range(L):
        prior = _ring_after(k, v, c, S, W)
        got = prefill_attention_prior(q[c:], k[c:], v[c:], prior, S, W)
        np.testing.assert_allclose(got, dense[c:], atol=1e-12)


def test_chunk_over_ring_built_in_pieces():
    """The prior ring's history (its head after wrapping) does not matter: a ring
    filled by chunks of 1, 5, 3 and 4 tokens gives the same result as one filled at once."""
    S, W, L, c = 2, 6, 30, 13
    q, k, v = _qkv(L, 4, 2, 8, 12)
    a = prefill_attention_prior(q[c:], k[c:], v[c:], _ring_after(k, v, c, S, W), S, W)
    ring = _ring_after(k, v, c, S, W, chunks=[1, 5, 3, 4])
    assert ring.head != _ring_after(k, v, c, S, W).head
    b = prefill_attention_prior(q[c:], k[c:], v[c:], ring, S, W)
    np.testing.assert_allclose(a, b, atol=1e-12)


def test_chunk_over_global_prefix_is_causal_attention():
    L, c, Hq, Hkv, D = 19, 8, 4, 4, 16
    q, k, v = _qkv(L, Hq, Hkv, D, 13)
    g = GlobalCache(64)
    g.append([(k[i], v[i]) for i in range(c)])
    got = prefill_attention_prior(q[c:], k[c:], v[c:], g, 0, None)
    causal = np.tril(np.ones((L, L), dtype=bool))
    np.testing.assert_allclose(got, _sdpa_rows(q, k, v, causal)[c:], atol=1e-12)


def test_empty_prior_is_the_chunk_alone():
    q, k, v = _qkv(12, 4, 2, 8, 14)
    np.testing.assert_allclose(prefill_attention_prior(q, k, v, RingCache(2, 5), 2, 5),
                               prefill_attention(q, k, v, 0, 2, 5), atol=1e-15)
    np.testing.assert_allclose(prefill_attention_prior(q, k, v, GlobalCache(32), 0, None),
                               prefill_attention(q, k, v, 0, 0, None), atol=1e-15)


def test_one_token_chunk_is_a_decode_step():
    """A chunk of one token at P equals the decode step at P (append, then attend over
    the cache's chronological rows)."""
    S, W, L = 3, 7, 20
    q, k, v = _qkv(L, 8, 2, 16, 15)
    for P in (0, 2, 9, 19):
        prior = _ring_after(k, v, P, S, W)
        got = prefill_attention_prior(q[P:P + 1], k[P:P + 1], v[P:P + 1], prior, S, W)[0]
        prior.append([(k[P], v[P])])
        np.testing.assert_allclose(got, decode_attention(prior, q[P]), atol=1e-12)


def test_prior_that_dropped_visible_keys_is_an_error():
    """A ring narrower than the chunk's window no longer holds keys the chunk's first
    query must see."""
    q, k, v = _qkv(20, 4, 2, 8, 16)
    prior = _ring_after(k, v, 12, 2, 3)
    with pytest.raises(ValueError):
        prefill_attention_prior(q[12:], k[12:], v[12:], prior, 2, 6)
