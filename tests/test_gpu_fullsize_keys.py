"""GPU parity at the workloads' full sizes, sensitive to every single key.

At full size one key carries about 1/4096 (windowed layers) to 1/131073 (a global
layer at 128k) of the softmax weight, far less than the 2e-2 bf16 tolerance of the
random-input checks, so those cannot tell a key lost or read twice at a split-K block
boundary, a ring wrap, the sink slots or a window-edge tile.  These tests make each
key count:

* Probe queries q = 0.  Every score is then exactly 0 and the softmax gives each
  visible key the weight 1 / |V(P)| ("Attention Sink 与 Streaming KV Cache", the
  visible set: sinks and the recent window), so the output is the plain mean of the
  visible V rows.  V rows are sparse random signs in {-1, 0, +1}: the kernels sum them
  exactly in fp32 (small integers), divide once and round once to bf16, so the
  output must lie within half a bf16 ulp (plus 2^-22 relative) of the float64 mean.
  A key more or less moves a dimension by about 1 / |V(P)|, which is several ulps
  for most dimensions at these sizes (each test checks that it has that power).
* fp32 caches at the windowed size, against the 2e-5 fp32 tolerance, where one key's
  weight is about 2.4e-4: the key rows themselves (the scores) are compared too.
"""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import (GlobalCache, RingCache, RopeSpec, attend, decode_attention as o_decode,
                                  prefill_attention as o_prefill, prefill_attention_prior, rope_rotate,
                                  visible_positions)
from sink_kv_attention_gb300 import synth
from tests.test_gpu_rope_append_decode import BF16_ATTN_ATOL, F32_ATTN_ATOL, bf16_ulp, f64

pytestmark = pytest.mark.gpu

DENSITY = 0.125   # share of nonzero signs in a probe V row


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def assert_exact_mean(got, want, n_keys):
    """got (bf16 output, as float64) against the float64 mean of +-1/0 rows over
    n_keys visible keys: within half a bf16 ulp plus 2^-22 relative, plus 1e-12 for
    the float64 rounding of the oracle's weights 1/n (a mean of zero comes out as
    about 1e-19 there).  Also checks that the bound is below half of one key's share
    (1 / n_keys) in a good part of the dimensions, so that one key lost or
    duplicated cannot pass."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    tol = 0.5 * bf16_ulp(want) + np.abs(want) * 2.0 ** -22 + 1e-12
    bad = np.abs(got - want) > tol
    assert not bad.any(), (int(bad.sum()), float(np.abs(got - want)[bad].max()), float(1.0 / np.max(n_keys)))
    sees = tol < 0.5 / np.asarray(n_keys, dtype=np.float64)[..., None]
    assert sees.mean() > 0.3, float(sees.mean())


def _ring_mirror_from_inputs(S, W, pos, head, count, k_b, v_b):
    """Oracle ring cache for one sequence holding the given input contents (all
    slots) and state: k_b, v_b are [H_kv, C, D] float64."""
    ring = RingCache(S, W)
    ring.pos, ring.head, ring.count = int(pos), int(head), int(count)
    for s in range(S + W):
        ring.slots[s] = (k_b[:, s], v_b[:, s])
    return ring


def _ring_states(B, S, W, seed):
    """Ragged ring states produced by the oracle's own state machine: sequences of
    lengths from 1 (only a sink) through partial rings to long wrapped ones."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 3 * (S + W), B)
    lens[:6] = [1, S, S + 1, S + W - 1, S + W, S + W + 1]
    states = []
    for n in lens:
        rc = RingCache(S, W)
        rc.append([None] * int(n))
        states.append((rc.pos, rc.head, rc.count))
    return states


# ---------------------------------------------------------------------------
# Windowed decode step (B=32, H_q=32, H_kv=8, d_h=128, S=4, W=4092)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("state", ["workload", "ragged"])
def test_window_decode_probe_every_key_counts(sk, state):
    """bf16, the windowed decode step's shapes and split plan: q = 0 for every head,
    V rows sparse signs; after the one-token append the output is the exact mean of
    the visible V rows.  'workload': the full rings of the benchmark (random heads);
    'ragged': rings from 1 token to several wraps."""
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    tbl = sk.RopeTable(D, c["r"], c["theta"], c["pos_hi"] + 2)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 211)
    synth.fill_sparse_signs_(layer.v, 212, DENSITY)
    if state == "workload":
        pos, head, count = synth.window_state(13, B, W, c["pos_lo"], c["pos_hi"])
    else:
        st = _ring_states(B, S, W, 213)
        pos = torch.tensor([x[0] for x in st])
        head = torch.tensor([x[1] for x in st], dtype=torch.int32)
        count = torch.tensor([x[2] for x in st], dtype=torch.int32)
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    k_in, v_in = f64(layer.k), f64(layer.v)
    q = torch.zeros(B, 1, Hq, D, dtype=torch.bfloat16, device="cuda")
    k = synth.normal((B, 1, Hkv, D), 214, torch.bfloat16).cuda()
    v = synth.sparse_signs((B, 1, Hkv, D), 215, DENSITY).cuda()
    k_raw, v_raw = f64(k), f64(v)
    sk.kv_append(tbl, layer, q, k, v)
    out = f64(sk.decode_attention(layer, q[:, 0].contiguous()))
    assert layer.error_bits() == 0
    spec = RopeSpec(D, c["r"], c["theta"])
    zero_q = np.zeros((Hq, D))
    for b in range(B):
        P = int(pos[b])
        ring = _ring_mirror_from_inputs(S, W, P, head[b], count[b], k_in[b], v_in[b])
        kr = rope_rotate(k_raw[b], [P], spec.omega(), 1.0, D)
        ring.append([(kr[0], v_raw[b, 0])])
        assert (int(layer.pos[b]), int(layer.head[b]), int(layer.count[b])) == (ring.pos, ring.head, ring.count)
        n = len(visible_positions(P, S + W, S))
        assert len(ring.chronological_slots()) == n
        assert_exact_mean(out[b], o_decode(ring, zero_q), n)


def test_window_decode_fp32_full_size(sk):
    """The windowed decode step in fp32 (q, k, v and both caches): RoPE + append +
    attention for all 32 sequences against the oracle at the fp32 tolerance (2e-5),
    where one key's weight (about 2.4e-4) is visible."""
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    tbl = sk.RopeTable(D, c["r"], c["theta"], c["pos_hi"] + 2)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=torch.float32,
                                v_dtype=torch.float32)
    synth.fill_normal_(layer.k, 221)
    synth.fill_normal_(layer.v, 222)
    pos, head, count = synth.window_state(223, B, W, c["pos_lo"], c["pos_hi"])
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    k_in, v_in = f64(layer.k), f64(layer.v)
    q = synth.normal((B, 1, Hq, D), 224).cuda()
    k = synth.normal((B, 1, Hkv, D), 225).cuda()
    v = synth.normal((B, 1, Hkv, D), 226).cuda()
    q_raw, k_raw, v_raw = f64(q), f64(k), f64(v)
    sk.kv_append(tbl, layer, q, k, v)
    out = f64(sk.decode_attention(layer, q[:, 0].contiguous()))
    assert layer.error_bits() == 0
    spec = RopeSpec(D, c["r"], c["theta"])
    worst = 0.0
    for b in range(B):
        P = int(pos[b])
        ring = _ring_mirror_from_inputs(S, W, P, head[b], count[b], k_in[b], v_in[b])
        qr = rope_rotate(q_raw[b], [P], spec.omega(), 1.0, D)
        kr = rope_rotate(k_raw[b], [P], spec.omega(), 1.0, D)
        ring.append([(kr[0], v_raw[b, 0])])
        worst = max(worst, float(np.abs(out[b] - o_decode(ring, qr[0])).max()))
    assert worst <= F32_ATTN_ATOL, worst


# ---------------------------------------------------------------------------
# Hybrid decode (B=16, global prefix 131072, sliding S=4 + W=4096)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["global", "sliding"])
def test_hybrid_layer_probe_every_key_counts(sk, kind):
    """One layer of the Llama-3-8B-shaped hybrid decode at full size (B=16, H_q=32,
    H_kv=8, d_h=128): a global layer holding a 131,072-token prefix, or a sliding
    layer (S=4, W=4096, full rings at random heads).  q = 0, V sparse signs: each
    output is the exact mean of the sequence's visible V rows, 131,073 or 4,100 of
    them."""
    c = synth.HYBRID
    B, Hq, Hkv, D, S, W, prefix = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"], c["prefix"]
    nrep = Hq // Hkv
    tbl = sk.RopeTable(D, c["r"], c["theta"], prefix + 2)
    if kind == "global":
        layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, D, capacity=prefix + 1)
    else:
        layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
        layer.count.fill_(W)
        layer.head.copy_(synth.randint((B,), 231, 0, W).to(torch.int32))
    synth.fill_normal_(layer.k, 232)
    synth.fill_sparse_signs_(layer.v, 233, DENSITY)
    layer.pos.fill_(prefix)
    head_in = layer.head.clone().cpu() if kind == "sliding" else None
    sample = [0, 7, 15] if kind == "global" else list(range(B))
    v_in = {b: layer.v[b].clone() for b in sample}
    q = torch.zeros(B, 1, Hq, D, dtype=torch.bfloat16, device="cuda")
    k = synth.normal((B, 1, Hkv, D), 234, torch.bfloat16).cuda()
    v = synth.sparse_signs((B, 1, Hkv, D), 235, DENSITY).cuda()
    v_raw = f64(v)
    sk.kv_append(tbl, layer, q, k, v)
    out = f64(sk.decode_attention(layer, q[:, 0].contiguous()))
    assert layer.error_bits() == 0
    assert layer.pos.tolist() == [prefix + 1] * B
    zero_q = np.zeros((nrep, D))
    for b in sample:
        vb = v_in[b]
        if kind == "global":
            slots = list(range(prefix))                        # the prefix, then the new row at slot prefix
            n = prefix + 1
        else:
            ring = RingCache(S, W)
            ring.pos, ring.head, ring.count = prefix, int(head_in[b]), W
            for s in range(S + W):
                ring.slots[s] = s
            ring.append([-1])                                  # the new row; -1 marks it
            slots = [s for s in ring.chronological_rows() if s >= 0]
            n = len(ring.chronological_rows())
            assert n == len(visible_positions(prefix, S + W, S))
        for g in range(Hkv):
            vals = f64(vb[g][slots])                           # [n-1, D]
            vals = np.concatenate([vals, v_raw[b, 0, g][None]])[:, None, :]
            keys = np.zeros_like(vals)                         # q = 0: keys do not enter
            want = attend(zero_q, keys, vals)
            assert_exact_mean(out[b, g * nrep:(g + 1) * nrep], want, n)


# ---------------------------------------------------------------------------
# Prefill chunk (T=32768, H_q=32, H_kv=8, d_h=128, S=4, W=4092)
# ---------------------------------------------------------------------------

def _interval_means(vpos, intervals):
    """Mean of vpos rows over a union of position intervals per query: vpos is
    [n_pos, H, D] float64 (exact small integers), intervals a list per query of
    (lo, hi) half-open ranges.  Returns ([T, H, D] means, [T] key counts)."""
    csum = np.concatenate([np.zeros((1,) + vpos.shape[1:]), np.cumsum(vpos, axis=0)])
    T = len(intervals)
    out = np.zeros((T,) + vpos.shape[1:])
    cnt = np.zeros(T)
    for t, iv in enumerate(intervals):
        for lo, hi in iv:
            out[t] += csum[hi] - csum[lo]
            cnt[t] += hi - lo
        out[t] /= cnt[t]
    return out, cnt


def test_prefill_probe_every_key_counts_full_chunk(sk):
    """The prefill workload (B=1, T=32768, S=4, W=4092, C=4096): q heads h % 4 == 0
    are probes (q = 0), the others random; V sparse signs.  Every row of every probe
    head is the exact mean of V over its visible positions (sinks 0..3 and the last
    4092 positions up to itself); random heads are checked on sampled rows at the bf16
    tolerance."""
    c = synth.PREFILL
    B, T, Hq, Hkv, D, S, W = c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    C = S + W
    nrep = Hq // Hkv
    q = synth.normal((B, T, Hq, D), 241, torch.bfloat16, device="cuda")
    q[:, :, ::nrep] = 0.0
    k = synth.normal((B, T, Hkv, D), 242, torch.bfloat16, device="cuda")
    v = torch.empty(B, T, Hkv, D, dtype=torch.bfloat16, device="cuda")
    synth.fill_sparse_signs_(v, 243, DENSITY)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = sk.prefill_attention(q, k, v, 0, S, W, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    v_in = f64(v[0])                                           # [T, Hkv, D]
    # visible sets as unions of intervals; checked against the oracle's V(P) on samples
    intervals = [[(0, t + 1)] if t < C else [(0, S), (t - W + 1, t + 1)] for t in range(T)]
    rng = np.random.default_rng(244)
    sample = sorted(set([0, 1, 3, 4, 5, 63, 64, 127, 128, 4090, 4091, 4092, 4095, 4096, 4097, 4223, 8191, 8192,
                         T - 129, T - 128, T - 1] + rng.integers(0, T, 24).tolist()))
    for t in sample:
        assert sorted(p for lo, hi in intervals[t] for p in range(lo, hi)) == visible_positions(t, C, S)
    want, cnt = _interval_means(v_in, intervals)               # [T, Hkv, D]
    got = f64(out[0, :, ::nrep])                               # probe heads: one per kv head
    assert_exact_mean(got, want, cnt[:, None])
    # the oracle itself on sampled rows, all heads
    o = o_prefill(f64(q[0]), f64(k[0]), v_in, 0, S, W, rows=sample)
    np.testing.assert_allclose(o[:, ::nrep], want[sample], rtol=0, atol=1e-12)
    got_s = f64(out[0, sample])
    rand_heads = [h for h in range(Hq) if h % nrep]
    assert float(np.abs(got_s[:, rand_heads] - o[:, rand_heads]).max()) <= BF16_ATTN_ATOL


def test_prefill_over_prior_ring_probe_every_key_counts(sk):
    """A second chunk of the prefill workload's shapes (2048 tokens at p0 = 32768) over
    a full ring wrapped at head 1234: probe heads q = 0, V sparse signs in the ring
    and the chunk.  Every row of every probe head is the exact mean over the ring's
    sinks, the ring's recent keys the row still sees, and the chunk up to itself."""
    B, Hq, Hkv, D, S, W, p0, T = 1, 32, 8, 128, 4, 4092, 32768, 2048
    nrep = Hq // Hkv
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 251)
    synth.fill_sparse_signs_(layer.v, 252, DENSITY)
    layer.pos.fill_(p0)
    layer.count.fill_(W)
    layer.head.fill_(1234)
    q = synth.normal((B, T, Hq, D), 253, torch.bfloat16, device="cuda")
    q[:, :, ::nrep] = 0.0
    k = synth.normal((B, T, Hkv, D), 254, torch.bfloat16, device="cuda")
    v = synth.sparse_signs((B, T, Hkv, D), 255, DENSITY).cuda()
    k_ring, v_ring = f64(layer.k[0]), f64(layer.v[0])
    out = sk.prefill_attention(q, k, v, p0, S, W, prior=layer, err=layer.err)
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    # the oracle's mirror of the prior ring: sinks at slots 0..3, recent positions
    # p0 - W .. p0 - 1 from the head on
    prior = RingCache(S, W)
    for s in range(S):
        prior.slots[s] = (k_ring[:, s], v_ring[:, s])
        prior.slot_pos[s] = s
    for ci in range(W):
        phys = (1234 + ci) % W
        prior.slots[S + phys] = (k_ring[:, S + phys], v_ring[:, S + phys])
        prior.slot_pos[S + phys] = p0 - W + ci
    prior.pos, prior.head, prior.count = p0, 1234, W
    # V by position over [p0 - W, p0 + T), the sinks separately
    vrec = np.stack([prior.slots[s][1] for s in prior.chronological_slots()[S:]] + list(f64(v[0])))
    sinks = np.stack([prior.slots[s][1] for s in range(S)])
    vpos = np.concatenate([sinks, vrec])                       # index: sinks, then position - (p0 - W) + S
    base = p0 - W
    intervals = [[(0, S), (P - W + 1 - base + S, P + 1 - base + S)] for P in range(p0, p0 + T)]
    want, cnt = _interval_means(vpos, intervals)
    got = f64(out[0, :, ::nrep])
    assert_exact_mean(got, want, cnt[:, None])
    rows = [0, 1, 127, 128, 1000, 2046, 2047]
    o = prefill_attention_prior(f64(q[0]), f64(k[0]), f64(v[0]), prior, S, W, rows=rows)
    np.testing.assert_allclose(o[:, ::nrep], want[rows], rtol=0, atol=1e-12)
    rand_heads = [h for h in range(Hq) if h % nrep]
    assert float(np.abs(f64(out[0, rows])[:, rand_heads] - o[:, rand_heads]).max()) <= BF16_ATTN_ATOL
