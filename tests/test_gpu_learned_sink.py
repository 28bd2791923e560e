"""GPU parity: learned per-head sink logits (a denominator-only softmax term, clamped
to [-10, 15]) in split-K decode and tensor-core prefill, against the float64 oracle."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import GlobalCache, RingCache, decode_attention as o_decode
from oracle.sinkkv_oracle import prefill_attention as o_prefill
from tests.test_gpu_rope_append_decode import BF16_ATTN_ATOL, F32_ATTN_ATOL, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def _sink_logits(Hq, seed):
    """Per-head logits over [-14, 19] (both clamp bounds crossed), shuffled."""
    from sink_kv_attention_gb300 import synth
    z = torch.linspace(-14.0, 19.0, Hq)
    return z[torch.randperm(Hq, generator=synth.generator(seed, "cpu"))].contiguous()


def _filled_ring(sk, B, Hkv, D, S, W, dtype, seed, pos_lo, pos_hi):
    from sink_kv_attention_gb300 import synth
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=dtype, v_dtype=dtype)
    synth.fill_normal_(layer.k, seed)
    synth.fill_normal_(layer.v, seed + 1)
    pos, head, count = synth.window_state(seed + 2, B, W, pos_lo, pos_hi)
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    return layer, pos, head, count


def _oracle_ring(S, W, pos, head, count, k_b, v_b):
    ring = RingCache(S, W)
    ring.pos, ring.head, ring.count = int(pos), int(head), int(count)
    for s in range(S + W):
        ring.slots[s] = (k_b[:, s], v_b[:, s])
    return ring


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,Hq,Hkv,D,S,W", [
    (3, 8, 2, 128, 4, 300),     # several units, each split over a few blocks
    (1, 4, 1, 128, 4, 4092),    # one unit split over every block of the grid
    (2, 16, 2, 64, 2, 200),     # head_dim 64, n_rep 8
    (2, 4, 4, 128, 0, 97),      # MHA, no pinned sinks
])
def test_ring_decode_with_learned_sinks(sk, dtype, B, Hq, Hkv, D, S, W):
    from sink_kv_attention_gb300 import synth
    layer, pos, head, count = _filled_ring(sk, B, Hkv, D, S, W, dtype, 100, W + S + 1, 3 * (W + S))
    q = synth.normal((B, Hq, D), 104, dtype).cuda()
    z = _sink_logits(Hq, 105)
    out = f64(sk.decode_attention(layer, q, sink_logits=z.cuda()))
    plain = f64(sk.decode_attention(layer, q))
    k_in, v_in = f64(layer.k), f64(layer.v)
    tol = F32_ATTN_ATOL if dtype == torch.float32 else BF16_ATTN_ATOL
    for b in range(B):
        ring = _oracle_ring(S, W, pos[b], head[b], count[b], k_in[b], v_in[b])
        want = o_decode(ring, f64(q[b]), sink_logits=z.numpy())
        np.testing.assert_allclose(out[b], want, rtol=0, atol=tol)
        np.testing.assert_allclose(plain[b], o_decode(ring, f64(q[b])), rtol=0, atol=tol)
    assert layer.error_bits() == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_global_decode_with_learned_sinks_and_short_sequences(sk, dtype):
    """Global layer with lengths 1 (a single key: a sigmoid gate), 2 and 700."""
    from sink_kv_attention_gb300 import synth
    B, Hq, Hkv, D = 3, 8, 2, 128
    layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, D, capacity=1024, k_dtype=dtype, v_dtype=dtype)
    synth.fill_normal_(layer.k, 110)
    synth.fill_normal_(layer.v, 111)
    lens = [1, 2, 700]
    layer.pos.copy_(torch.tensor(lens, dtype=torch.int64))
    q = synth.normal((B, Hq, D), 112, dtype).cuda()
    z = _sink_logits(Hq, 113)
    out = f64(sk.decode_attention(layer, q, sink_logits=z.cuda()))
    k_in, v_in = f64(layer.k), f64(layer.v)
    tol = F32_ATTN_ATOL if dtype == torch.float32 else BF16_ATTN_ATOL
    for b in range(B):
        g = GlobalCache(1024)
        g.append([(k_in[b][:, t], v_in[b][:, t]) for t in range(lens[b])])
        np.testing.assert_allclose(out[b], o_decode(g, f64(q[b]), sink_logits=z.numpy()), rtol=0, atol=tol)


def test_noalloc_decode_with_learned_sinks_matches_workspace_call(sk):
    from sink_kv_attention_gb300 import synth
    layer, _, _, _ = _filled_ring(sk, 4, 8, 128, 4, 1000, torch.bfloat16, 120, 1100, 5000)
    q = synth.normal((4, 32, 128), 124, torch.bfloat16).cuda()
    z = _sink_logits(32, 125).cuda()
    want = sk.decode_attention(layer, q, sink_logits=z)
    got = sk.decode_attention_noalloc(layer, q, torch.empty_like(q), sink_logits=z)
    assert torch.equal(got, want)


def test_window_decode_full_size_with_learned_sinks_sampled(sk):
    """The windowed decode step's shapes (B=32, H_q=32, H_kv=8, d_h=128, S=4, W=4092)
    with learned sinks; 6 sequences checked against the oracle."""
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    layer, pos, head, count = _filled_ring(sk, B, Hkv, D, S, W, torch.bfloat16, 130, c["pos_lo"], c["pos_hi"])
    q = synth.normal((B, Hq, D), 134, torch.bfloat16).cuda()
    z = _sink_logits(Hq, 135)
    out = f64(sk.decode_attention(layer, q, sink_logits=z.cuda()))
    for b in [0, 5, 13, 21, 30, 31]:
        ring = _oracle_ring(S, W, pos[b], head[b], count[b], f64(layer.k[b]), f64(layer.v[b]))
        want = o_decode(ring, f64(q[b]), sink_logits=z.numpy())
        np.testing.assert_allclose(out[b], want, rtol=0, atol=BF16_ATTN_ATOL)


@pytest.mark.parametrize("T,S,W,p0", [
    (300, 4, 100, 0),
    (257, 4, 0, 0),      # global layer
    (513, 3, 130, 1),
    (1, 4, 16, 0),       # one token: the sink against a single key
])
def test_prefill_with_learned_sinks_all_rows(sk, T, S, W, p0):
    from sink_kv_attention_gb300 import synth
    B, Hq, Hkv, D = 2, 8, 2, 128
    q = synth.normal((B, T, Hq, D), 140, torch.bfloat16).cuda()
    k = synth.normal((B, T, Hkv, D), 141, torch.bfloat16).cuda()
    v = synth.normal((B, T, Hkv, D), 142, torch.bfloat16).cuda()
    z = _sink_logits(Hq, 143)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = f64(sk.prefill_attention(q, k, v, p0, S, W, err=err, sink_logits=z.cuda()))
    assert int(err.item()) == 0
    for b in range(B):
        want = o_prefill(f64(q[b]), f64(k[b]), f64(v[b]), p0, S, W if W > 0 else None, sink_logits=z.numpy())
        worst = float(np.abs(out[b] - want).max())
        assert worst <= BF16_ATTN_ATOL, (b, worst)


def test_learned_sink_arguments_are_checked(sk):
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, 1, 128, sinks=1, window=8)
    q = torch.zeros(1, 4, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        sk.decode_attention(layer, q, sink_logits=torch.zeros(3, device="cuda"))
    with pytest.raises(ValueError):
        sk.decode_attention(layer, q, sink_logits=torch.zeros(4, dtype=torch.float64, device="cuda"))
