"""GPU parity: tensor-core prefill of a chunk that continues a cached sequence (the
chunk attends over the keys a ring or global cache holds for positions before p0 and
over itself), against the float64 oracle."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import (GlobalCache, RingCache, RopeSpec, prefill_attention_prior, rope_rotate)
from sink_kv_attention_gb300 import synth
from tests.test_gpu_rope_append_decode import BF16_ATTN_ATOL, f64

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def _ring_mirror(layer, b, S, W, p0, head, count):
    """The oracle's RingCache holding sequence b of a device ring layer as given:
    the same slots, state and slot positions (O4's layout for a cache at p0)."""
    rc = RingCache(S, W)
    k = f64(layer.k[b])   # [Hkv, C, D]
    v = f64(layer.v[b])
    s0 = min(S, p0)
    for s in range(s0):
        rc.slots[s] = (k[:, s], v[:, s])
        rc.slot_pos[s] = s
    for ci in range(count):
        phys = (head + ci) % W if count == W else ci
        rc.slots[S + phys] = (k[:, S + phys], v[:, S + phys])
        rc.slot_pos[S + phys] = p0 - count + ci
    rc.pos, rc.head, rc.count = p0, head, count
    return rc


def _global_mirror(layer, b, p0):
    g = GlobalCache(layer.capacity)
    k, v = f64(layer.k[b]), f64(layer.v[b])
    g.append([(k[:, P], v[:, P]) for P in range(p0)])
    return g


def _chunk(B, T, Hq, Hkv, seed):
    q = synth.normal((B, T, Hq, D), seed, torch.bfloat16)
    k = synth.normal((B, T, Hkv, D), seed + 1, torch.bfloat16)
    v = synth.normal((B, T, Hkv, D), seed + 2, torch.bfloat16)
    return q, k, v


def _check(sk, layer, mirrors, q, k, v, p0, S, W, rows=None, sink_logits=None):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    z = None if sink_logits is None else sink_logits.cuda()
    out = f64(sk.prefill_attention(qd, kd, vd, p0, S, W, prior=layer, err=layer.err, sink_logits=z))
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    T = q.shape[1]
    rows = list(range(T)) if rows is None else rows
    zn = None if sink_logits is None else sink_logits.numpy()
    for b, prior in enumerate(mirrors):
        want = prefill_attention_prior(f64(q[b]), f64(k[b]), f64(v[b]), prior, S, W if W > 0 else None,
                                       rows=rows, sink_logits=zn)
        np.testing.assert_allclose(out[b][rows], want, rtol=0, atol=BF16_ATTN_ATOL)


@pytest.mark.parametrize("p0,T,S,W,Hq,Hkv", [
    (2, 300, 4, 100, 8, 2),      # the prior holds only sink positions 0, 1
    (50, 300, 4, 100, 8, 2),     # ring not yet full (46 recent)
    (250, 300, 4, 100, 8, 2),    # ring full and wrapped at a different head per sequence
    (1000, 129, 0, 61, 4, 4),    # no sinks, MHA, a ragged chunk
    (700, 260, 3, 300, 16, 2),   # 8 q heads per CTA
])
def test_prefill_over_ring_prior_matches_oracle(sk, p0, T, S, W, Hq, Hkv):
    B = 2
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 21)
    synth.fill_normal_(layer.v, 22)
    count = min(W, p0 - min(S, p0))
    heads = [count % W if count < W else (37 * b + 11) % W for b in range(B)]
    layer.pos.fill_(p0)
    layer.count.fill_(count)
    layer.head.copy_(torch.tensor(heads, dtype=torch.int32))
    mirrors = [_ring_mirror(layer, b, S, W, p0, heads[b], count) for b in range(B)]
    q, k, v = _chunk(B, T, Hq, Hkv, 30)
    _check(sk, layer, mirrors, q, k, v, p0, S, W)


@pytest.mark.parametrize("p0,T,S,W", [
    (300, 200, 0, 0),     # causal over the whole prefix
    (300, 200, 4, 100),   # sinks + window over a global cache
    (5, 140, 4, 0),
])
def test_prefill_over_global_prior_matches_oracle(sk, p0, T, S, W):
    B, Hq, Hkv = 2, 8, 2
    layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, D, capacity=512)
    synth.fill_normal_(layer.k, 23)
    synth.fill_normal_(layer.v, 24)
    layer.pos.fill_(p0)
    mirrors = [_global_mirror(layer, b, p0) for b in range(B)]
    q, k, v = _chunk(B, T, Hq, Hkv, 40)
    _check(sk, layer, mirrors, q, k, v, p0, S, W)


def test_prefill_prior_with_learned_sinks(sk):
    B, Hq, Hkv, S, W, p0, T = 1, 8, 2, 4, 100, 400, 200
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 25)
    synth.fill_normal_(layer.v, 26)
    layer.pos.fill_(p0)
    layer.count.fill_(W)
    layer.head.fill_(17)
    mirrors = [_ring_mirror(layer, 0, S, W, p0, 17, W)]
    q, k, v = _chunk(B, T, Hq, Hkv, 50)
    _check(sk, layer, mirrors, q, k, v, p0, S, W, sink_logits=torch.linspace(-12.0, 16.0, Hq))


def test_chunked_prefill_through_the_library(sk):
    """A prompt in three chunks.  The first is rotated and appended by kv_append.  Each
    later chunk is rotated by rope_apply, attends over the ring the earlier chunks left,
    and is then appended as given (kv_append without a table).  Rows, ring state and
    cached keys match the oracle's chunked prefill of the raw prompt rotated in
    float64."""
    B, Hq, Hkv, S, W = 2, 8, 2, 4, 150
    chunks = [333, 260, 97]
    L = sum(chunks)
    spec = RopeSpec(D, D, 1e4)
    tbl = sk.RopeTable(D, D, 1e4, L + 8)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    q, k, v = _chunk(B, L, Hq, Hkv, 60)
    kr = [rope_rotate(f64(k[b]), range(L), spec.omega(), 1.0, D) for b in range(B)]
    rings = [RingCache(S, W) for _ in range(B)]
    sk.kv_append(tbl, layer, None, k[:, :chunks[0]].contiguous().cuda(), v[:, :chunks[0]].contiguous().cuda())
    for b in range(B):
        rings[b].append([(kr[b][P], f64(v[b, P])) for P in range(chunks[0])])
    p0 = chunks[0]
    for T in chunks[1:]:
        qc, kc = q[:, p0:p0 + T].contiguous().cuda(), k[:, p0:p0 + T].contiguous().cuda()
        vc = v[:, p0:p0 + T].contiguous().cuda()
        posn = torch.arange(p0, p0 + T, dtype=torch.int64, device="cuda").repeat(B)
        sk.rope_apply(tbl, qc.view(B * T, Hq, D), posn)
        sk.rope_apply(tbl, kc.view(B * T, Hkv, D), posn)
        out = f64(sk.prefill_attention(qc, kc, vc, p0, S, W, prior=layer, err=layer.err))
        sk.kv_append(None, layer, None, kc, vc)
        torch.cuda.synchronize()
        assert layer.error_bits() == 0
        rows = sorted({0, 1, 63, 64, T // 2, T - 1})
        for b in range(B):
            qr = rope_rotate(f64(q[b, p0:p0 + T]), range(p0, p0 + T), spec.omega(), 1.0, D)
            want = prefill_attention_prior(qr, kr[b][p0:p0 + T], f64(v[b, p0:p0 + T]), rings[b], S, W, rows=rows)
            np.testing.assert_allclose(out[b][rows], want, rtol=0, atol=BF16_ATTN_ATOL)
            rings[b].append([(kr[b][P], f64(v[b, P])) for P in range(p0, p0 + T)])
        p0 += T
        # the append of rotated keys moved the state as the oracle's ring and copied the
        # keys bit for bit
        assert layer.pos.tolist() == [p0] * B
        assert layer.head.tolist() == [r.head for r in rings]
        assert layer.count.tolist() == [r.count for r in rings]
        kcache = layer.k.cpu()
        for b in range(B):
            for s_ in range(S + W):
                P = rings[b].slot_pos[s_]
                if P >= p0 - T:  # a key of this chunk
                    assert torch.equal(kcache[b, :, s_], kc[b, P - (p0 - T)].cpu())


def test_prior_state_mismatch_sets_error_bit(sk):
    """A ring whose pos does not match p0 sets SK_DEVERR_STATE (reads stay in the cache)."""
    B, Hq, Hkv, S, W, p0, T = 1, 8, 2, 4, 100, 250, 64
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    layer.pos.fill_(p0 + 3)
    layer.count.fill_(W)
    q, k, v = _chunk(B, T, Hq, Hkv, 70)
    sk.prefill_attention(q.cuda(), k.cuda(), v.cuda(), p0, S, W, prior=layer, err=layer.err)
    torch.cuda.synchronize()
    assert layer.error_bits() & sk.SK_DEVERR_STATE
    status, bits = sk.sync_check(layer.err, clear=True)
    assert status == sk.SK_ERR_ARG and bits & sk.SK_DEVERR_STATE
    assert layer.error_bits() == 0


def test_prefill_prior_at_windowed_sizes_sampled(sk):
    """The prefill workload's shapes (H_q=32, H_kv=8, S=4, W=4092) for a second chunk
    of 2048 tokens at p0 = 32768 over a full, wrapped ring; sampled rows."""
    B, Hq, Hkv, S, W, p0, T = 1, 32, 8, 4, 4092, 32768, 2048
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 27)
    synth.fill_normal_(layer.v, 28)
    layer.pos.fill_(p0)
    layer.count.fill_(W)
    layer.head.fill_(1234)
    mirrors = [_ring_mirror(layer, 0, S, W, p0, 1234, W)]
    q, k, v = _chunk(B, T, Hq, Hkv, 80)
    _check(sk, layer, mirrors, q, k, v, p0, S, W, rows=[0, 1, 127, 128, 1000, 2046, 2047])
