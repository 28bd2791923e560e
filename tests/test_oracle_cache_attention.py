"""Pins of the oracle's ring/global caches, visible sets and attention."""
import itertools

import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import (CapacityError, GlobalCache, RingCache, attend, decode_attention,
                                  mask_allows, prefill_attention, visible_positions)
from tests.conftest import golden_path


def _golden_table():
    rows = {}
    with open(golden_path("visible_c6_s2_t10.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            i, vis = line.split(":")
            rows[int(i)] = [int(x) for x in vis.split(",")]
    return rows


def test_visible_table_closed_form():
    table = _golden_table()
    assert sorted(table) == list(range(10))
    for i, vis in table.items():
        assert visible_positions(i, 6, 2) == vis
    assert [len(table[i]) for i in range(10)] == [1, 2, 3, 4, 5, 6, 6, 6, 6, 6]
    assert table[9] == [0, 1, 6, 7, 8, 9]


def test_visible_table_from_ring_state_machine():
    """Appending one token at a time into S=2 sinks + a ring of W=4 holds exactly
    the page's visible positions after every step."""
    table = _golden_table()
    c = RingCache(2, 4)
    for i in range(10):
        c.append([("tok", i)])
        assert c.chronological_positions() == table[i]
        assert c.pos == i + 1
        assert [r[1] for r in c.chronological_rows()] == table[i]


def test_ring_rollover_order_window3():
    """7 tokens into a window-3 ring read back as [5, 6, 7]; the length caps at the
    window ("KV-Cache Engineering", 6: the rollover-order and append-windowed tests)."""
    c = RingCache(0, 3)
    for v in range(1, 8):
        c.append([v])
        assert c.count == min(v, 3)
    assert c.chronological_rows() == [5, 6, 7]
    one_shot = RingCache(0, 3)
    one_shot.append(list(range(1, 8)))          # T_new >= window: keep the last window
    assert one_shot.chronological_rows() == [5, 6, 7]
    assert (one_shot.head, one_shot.count) == (0, 3)
    short = RingCache(0, 5)
    short.append([1, 2, 3])                     # T_new < window: fill from 0
    assert (short.head, short.count) == (3, 3) and short.slots[:3] == [1, 2, 3]


def test_ring_brute_force_all_chunkings():
    """For all S, W with S + W <= 12 and random chunkings of up to 40 tokens, the ring
    holds exactly V(last position) in chronological order after every append."""
    rng = np.random.default_rng(0)
    for S in range(0, 5):
        for W in range(1, 13 - S):
            C = S + W
            for _ in range(4):
                c = RingCache(S, W)
                T = int(rng.integers(1, 41))
                done = 0
                while done < T:
                    n = int(rng.integers(1, 2 * W + 3))
                    n = min(n, T - done)
                    c.append([done + t for t in range(n)])
                    done += n
                    assert c.chronological_positions() == visible_positions(done - 1, C, S)
                    assert c.chronological_rows() == visible_positions(done - 1, C, S)
                    assert 0 <= c.head < W and 0 <= c.count <= W
                    # never wrapped <=> head == count
                    if c.count < W:
                        assert c.head == c.count


def test_mask_rule_equals_visible_set():
    for S, W in [(0, 3), (2, 4), (4, 9), (1, 1)]:
        for P in range(40):
            ks = [k for k in range(P + 1) if mask_allows(P, k, S, W)]
            assert ks == visible_positions(P, S + W, S)
        assert [k for k in range(9) if mask_allows(8, k, S, None)] == list(range(9))


def test_global_cache_capacity_is_loud():
    g = GlobalCache(5)
    g.append([0, 1, 2])
    g.append([3, 4])
    assert g.chronological_positions() == [0, 1, 2, 3, 4]
    with pytest.raises(CapacityError):
        g.append([5])
    assert g.pos == 5


def _sdpa(q, k, v, mask):
    """torch's float64 CPU scaled_dot_product_attention with kv heads broadcast;
    q [T,Hq,D], k/v [T,Hkv,D], mask [T,T] bool (True = attend)."""
    n_rep = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(n_rep, 0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(n_rep, 0)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(mask))
    return o.permute(1, 0, 2).numpy()


def _qkv(T, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, Hq, D)), rng.standard_normal((T, Hkv, D)),
            rng.standard_normal((T, Hkv, D)))


def test_dense_mask_attention_matches_library_sdpa():
    """The page's C=6, S=2 table as a boolean mask through torch's SDPA."""
    table = _golden_table()
    q, k, v = _qkv(10, 8, 4, 64, 1)
    mask = np.zeros((10, 10), dtype=bool)
    for i, vis in table.items():
        mask[i, vis] = True
    np.testing.assert_allclose(prefill_attention(q, k, v, 0, 2, 4), _sdpa(q, k, v, mask), atol=1e-12)


def test_special_cases_reduce_to_textbook_attention():
    q, k, v = _qkv(24, 4, 2, 16, 2)
    causal = np.tril(np.ones((24, 24), dtype=bool))
    # capacity larger than T: full causal attention
    np.testing.assert_allclose(prefill_attention(q, k, v, 0, 4, 60), _sdpa(q, k, v, causal), atol=1e-12)
    # global layer: full causal
    np.testing.assert_allclose(prefill_attention(q, k, v, 0, 0, None), _sdpa(q, k, v, causal), atol=1e-12)
    # S = 0: a pure sliding window of 5
    band = causal & (np.arange(24)[:, None] - np.arange(24)[None, :] < 5)
    np.testing.assert_allclose(prefill_attention(q, k, v, 0, 0, 5), _sdpa(q, k, v, band), atol=1e-12)
    # sink + window differs from full causal past the capacity (page 4: "> 1e-3")
    sw = prefill_attention(q, k, v, 0, 2, 4)
    full = prefill_attention(q, k, v, 0, 0, None)
    assert np.abs(sw[6:] - full[6:]).max() > 1e-3


def test_zero_query_gives_uniform_average_of_visible_values():
    rng = np.random.default_rng(3)
    keys = rng.standard_normal((9, 2, 8))
    vals = rng.standard_normal((9, 2, 8))
    out = attend(np.zeros((4, 8)), keys, vals)
    np.testing.assert_allclose(out[0], vals[:, 0].mean(0), atol=1e-15)
    np.testing.assert_allclose(out[3], vals[:, 1].mean(0), atol=1e-15)


@pytest.mark.parametrize("S,W", [(2, 4), (0, 3), (4, 5)])
def test_incremental_decode_equals_dense_sink_mask(S, W):
    """Token-by-token decode through the ring equals dense attention with the
    sink mask (page 4's incremental vs dense, 1e-12), with GQA 8:4."""
    T, Hq, Hkv, D = 17, 8, 4, 64
    q, k, v = _qkv(T, Hq, Hkv, D, 4)
    dense = prefill_attention(q, k, v, 0, S, W)
    c = RingCache(S, W)
    for t in range(T):
        c.append([(k[t], v[t])])
        np.testing.assert_allclose(decode_attention(c, q[t]), dense[t], atol=1e-12)


def test_global_decode_equals_causal():
    T, Hq, Hkv, D = 12, 4, 4, 32
    q, k, v = _qkv(T, Hq, Hkv, D, 5)
    dense = prefill_attention(q, k, v, 0, 0, None)
    g = GlobalCache(64)
    for t in range(T):
        g.append([(k[t], v[t])])
        np.testing.assert_allclose(decode_attention(g, q[t]), dense[t], atol=1e-12)


# ---- learned sink logits ---------------------------------------------------------------

def _sdpa_with_sink_column(q, k, v, z):
    """torch's float64 SDPA over the keys plus one extra key column whose logit is
    forced to z[h] by an additive mask (a zero key scores 0, the mask adds z[h]) and
    whose value row is zero: a per-head term exp(z_h) in the denominator only.
    q [Hq,D], k/v [n,Hkv,D]."""
    n_rep = q.shape[0] // k.shape[1]
    n, D = k.shape[0], k.shape[2]
    kt = torch.from_numpy(np.concatenate([k, np.zeros((1,) + k.shape[1:])])).permute(1, 0, 2)
    vt = torch.from_numpy(np.concatenate([v, np.zeros((1,) + v.shape[1:])])).permute(1, 0, 2)
    kt, vt = kt.repeat_interleave(n_rep, 0), vt.repeat_interleave(n_rep, 0)
    mask = torch.zeros(q.shape[0], 1, n + 1, dtype=torch.float64)
    mask[:, 0, n] = torch.from_numpy(np.asarray(z, dtype=np.float64))
    qt = torch.from_numpy(q)[:, None, :]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)[:, 0].numpy()


def test_learned_sink_equals_extra_zero_value_column_in_library_sdpa():
    """A learned sink is a per-head logit in the softmax denominator with no value
    ("RoPE, scaling, sliding window, attention sinks", "Hybrid models break the
    uniform-spec assumption"): the same as one more key column of logit z_h and value 0."""
    rng = np.random.default_rng(11)
    q, k, v = rng.standard_normal((8, 64)) * 2, rng.standard_normal((37, 4, 64)), rng.standard_normal((37, 4, 64))
    z = np.array([-9.5, -3.0, 0.0, 0.7, 2.5, 4.0, 9.0, 14.9])
    np.testing.assert_allclose(attend(q, k, v, z), _sdpa_with_sink_column(q, k, v, z), atol=1e-12)


def test_learned_sink_single_key_is_a_sigmoid_gate():
    """One visible key of logit s and value v: out = v * sigmoid(s - z)."""
    q = np.array([[2.0, 0.0, 0.0, 0.0]])
    k = np.array([[[1.5, 0.0, 0.0, 0.0]]])      # s = 2 * 1.5 / sqrt(4) = 1.5
    v = np.array([[[1.0, -2.0, 0.5, 3.0]]])
    out = attend(q, k, v, [0.5])
    np.testing.assert_allclose(out[0], v[0, 0] * 0.7310585786300049, rtol=1e-15)  # sigmoid(1)
    # equal logits: half the weight goes to the sink
    np.testing.assert_allclose(attend(q, k, v, [1.5])[0], v[0, 0] * 0.5, rtol=1e-15)


def test_learned_sink_logits_are_clamped_to_page_bounds():
    """The forward pass clamps the sink bias to [-10, 15] ("Inference & 128K Long
    Context", "Sink clamp cache")."""
    rng = np.random.default_rng(12)
    q, k, v = rng.standard_normal((4, 16)), rng.standard_normal((9, 2, 16)), rng.standard_normal((9, 2, 16))
    np.testing.assert_array_equal(attend(q, k, v, [100.0, -1e9, 15.0, -10.0]),
                                  attend(q, k, v, [15.0, -10.0, 15.0, -10.0]))
    # inside the bounds nothing is clamped: z = 14.99 differs from 15
    assert np.abs(attend(q, k, v, [14.99] * 4) - attend(q, k, v, [15.0] * 4)).max() > 1e-12


def test_learned_sink_shrinks_plain_attention_by_its_weight():
    """out_sink = (1 - p_sink) * out_plain with p_sink = e^z / (e^z + sum_j e^{s_j});
    the sum of exponentials is taken with an explicit loop."""
    rng = np.random.default_rng(13)
    q, k, v = rng.standard_normal((2, 8)), rng.standard_normal((5, 1, 8)), rng.standard_normal((5, 1, 8))
    z = [1.25, -4.0]
    got = attend(q, k, v, z)
    plain = attend(q, k, v)
    for h in range(2):
        tot = 0.0
        for j in range(5):
            tot += float(np.exp(sum(q[h, d] * k[j, 0, d] for d in range(8)) / np.sqrt(8)))
        p_sink = np.exp(z[h]) / (np.exp(z[h]) + tot)
        np.testing.assert_allclose(got[h], (1 - p_sink) * plain[h], rtol=1e-12, atol=1e-15)


def test_learned_sink_in_decode_and_prefill_agree():
    """A decode step at P equals row P of the prefill with the same mask and sinks."""
    T, Hq, Hkv, D, S, W = 13, 4, 2, 16, 2, 4
    q, k, v = _qkv(T, Hq, Hkv, D, 14)
    z = [-1.0, 0.5, 3.0, 20.0]
    dense = prefill_attention(q, k, v, 0, S, W, sink_logits=z)
    c = RingCache(S, W)
    for t in range(T):
        c.append([(k[t], v[t])])
        np.testing.assert_allclose(decode_attention(c, q[t], sink_logits=z), dense[t], atol=1e-12)
