"""GPU parity of decode attention at small batches, where one (sequence, kv head) unit
meets many split blocks and the combine gives each (sequence, q head) a group of warps:
1 sequence of 8 kv heads meets about 20 of the 152 blocks per unit (8 warps per head),
2 sequences about 10 (4 warps), 4 about 5 (2 warps); a single sequence with one kv head
(MQA) meets every block (8 warps, several batches of partials each)."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import RopeSpec, attend, decode_attention as o_decode, rope_rotate
from sink_kv_attention_gb300 import synth
from tests.test_gpu_fullsize_keys import DENSITY, _ring_mirror_from_inputs, assert_exact_mean
from tests.test_gpu_rope_append_decode import BF16_ATTN_ATOL, F32_ATTN_ATOL, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


@pytest.mark.parametrize("B", [1, 2, 3, 4, 6])
def test_small_batch_window_decode(sk, B):
    """The windowed decode step's shapes (H_q=32, H_kv=8, d_h=128, S=4, W=4092, full rings
    at random heads) at batch B: RoPE + append + attention.  Heads h % 4 == 0 are probes
    (q = 0, output the exact mean of the visible V rows, V sparse signs); the others are
    random and compared with the oracle at the bf16 tolerance."""
    c = synth.WINDOW
    Hq, Hkv, D, S, W = c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    nrep = Hq // Hkv
    tbl = sk.RopeTable(D, c["r"], c["theta"], c["pos_hi"] + 2)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 301 + B)
    synth.fill_sparse_signs_(layer.v, 302 + B, DENSITY)
    pos, head, count = synth.window_state(303 + B, B, W, c["pos_lo"], c["pos_hi"])
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    k_in, v_in = f64(layer.k), f64(layer.v)
    q = synth.normal((B, 1, Hq, D), 304 + B, torch.bfloat16).cuda()
    q[:, :, ::nrep] = 0.0
    k = synth.normal((B, 1, Hkv, D), 305 + B, torch.bfloat16).cuda()
    v = synth.sparse_signs((B, 1, Hkv, D), 306 + B, DENSITY).cuda()
    q_raw, k_raw, v_raw = f64(q), f64(k), f64(v)
    sk.kv_append(tbl, layer, q, k, v)
    out = f64(sk.decode_attention(layer, q[:, 0].contiguous()))
    assert layer.error_bits() == 0
    spec = RopeSpec(D, c["r"], c["theta"])
    rand = [h for h in range(Hq) if h % nrep]
    for b in range(B):
        P = int(pos[b])
        ring = _ring_mirror_from_inputs(S, W, P, head[b], count[b], k_in[b], v_in[b])
        qr = rope_rotate(q_raw[b], [P], spec.omega(), 1.0, D)
        kr = rope_rotate(k_raw[b], [P], spec.omega(), 1.0, D)
        ring.append([(kr[0], v_raw[b, 0])])
        want = o_decode(ring, qr[0])
        assert_exact_mean(out[b, ::nrep], want[::nrep], S + W)
        assert float(np.abs(out[b, rand] - want[rand]).max()) <= BF16_ATTN_ATOL


@pytest.mark.parametrize("n_keys", [20000, 1000, 153])
@pytest.mark.parametrize("Hq,D", [(4, 128), (8, 64)])
def test_single_sequence_mqa_global_fp32(sk, n_keys, Hq, D):
    """One sequence, one kv head (MQA), a global layer of n_keys fp32 rows: the unit meets
    every split block that holds one of its rows (up to 152), so each of the combine's 8
    warps per head folds several batches of partials.  fp32 tolerance."""
    layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, 1, D, capacity=n_keys, k_dtype=torch.float32,
                                v_dtype=torch.float32)
    synth.fill_normal_(layer.k, 311)
    synth.fill_normal_(layer.v, 312)
    layer.pos.fill_(n_keys)
    q = synth.normal((1, Hq, D), 313).cuda()
    out = f64(sk.decode_attention(layer, q))
    assert layer.error_bits() == 0
    keys, vals = f64(layer.k[0, 0]), f64(layer.v[0, 0])
    want = attend(f64(q[0]), keys[:, None, :], vals[:, None, :])
    np.testing.assert_allclose(out[0], want, rtol=0, atol=F32_ATTN_ATOL)


def test_single_sequence_learned_sinks(sk):
    """Learned sink logits through the grouped combine (one sequence of the windowed
    shapes): the sink term enters when the group's warps merge."""
    c = synth.WINDOW
    Hq, Hkv, D, S, W = c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 321)
    synth.fill_normal_(layer.v, 322)
    layer.pos.fill_(20000)
    layer.count.fill_(W)
    layer.head.fill_(777)
    q = synth.normal((1, Hq, D), 323, torch.bfloat16).cuda()
    z = torch.linspace(-12.0, 17.0, Hq)
    out = f64(sk.decode_attention(layer, q, sink_logits=z.cuda()))
    ring = _ring_mirror_from_inputs(S, W, 20000, 777, W, f64(layer.k[0]), f64(layer.v[0]))
    want = o_decode(ring, f64(q[0]), sink_logits=z.numpy())
    np.testing.assert_allclose(out[0], want, rtol=0, atol=BF16_ATTN_ATOL)
