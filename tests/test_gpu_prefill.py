"""GPU parity: tensor-core prefill attention (causal + window + sinks) and the prefill
append (RoPE + ring write of a long chunk), against the float64 oracle."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import RingCache, RopeSpec, prefill_attention as o_prefill, rope_rotate
from tests.test_gpu_rope_append_decode import BF16_ATTN_ATOL, assert_rows_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


@pytest.mark.parametrize("T,S,W,p0", [
    (300, 4, 100, 0),     # window shorter than a query block, ragged last block
    (300, 0, 100, 0),     # pure sliding window
    (300, 4, 0, 0),       # global layer: causal only
    (257, 4, 1000, 0),    # window longer than the chunk: full causal
    (513, 3, 130, 1),     # chunk starting at position 1: keys 0, 1 are sinks
    (64, 4, 16, 0),       # a single partial query block
    (1, 4, 16, 0),        # one token
])
def test_prefill_matches_oracle_all_rows(sk, T, S, W, p0):
    _prefill_case(sk, T, S, W, p0, 4, 2)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 1), (6, 2), (16, 2)])
def test_prefill_head_packing(sk, Hq, Hkv):
    """q heads of a GQA group packed into one CTA: 1 (MHA), 8 (16 queries per block),
    n_rep = 3 (no packing possible beyond 1), 8 of 8."""
    _prefill_case(sk, 300, 4, 100, 0, Hq, Hkv)


def _prefill_case(sk, T, S, W, p0, Hq, Hkv):
    from sink_kv_attention_gb300 import synth
    B, D = 2, 128
    q = synth.normal((B, T, Hq, D), 60, torch.bfloat16).cuda()
    k = synth.normal((B, T, Hkv, D), 61, torch.bfloat16).cuda()
    v = synth.normal((B, T, Hkv, D), 62, torch.bfloat16).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = f64(sk.prefill_attention(q, k, v, p0, S, W, err=err))
    assert int(err.item()) == 0
    for b in range(B):
        want = o_prefill(f64(q[b]), f64(k[b]), f64(v[b]), p0, S, W if W > 0 else None)
        worst = float(np.abs(out[b] - want).max())
        assert worst <= BF16_ATTN_ATOL, (b, worst)


def test_prefill_chunk_full_size_sampled(sk):
    """B=1, T=32768, H_q=32, H_kv=8, d_h=r=128, S=4, W=4092 (C=4096): RoPE is applied
    to Q and K and the rotated K/V written to the ring (only the last window kept),
    then attention of the chunk over itself; sampled rows against the oracle."""
    from sink_kv_attention_gb300 import synth
    c = synth.PREFILL
    B, T, Hq, Hkv, D, S, W = c["B"], c["T"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    tbl = sk.RopeTable(D, c["r"], c["theta"], T + 8)
    spec = RopeSpec(D, c["r"], c["theta"])
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    q = synth.normal((B, T, Hq, D), 63, torch.bfloat16, device="cuda")
    k = synth.normal((B, T, Hkv, D), 64, torch.bfloat16, device="cuda")
    v = synth.normal((B, T, Hkv, D), 65, torch.bfloat16, device="cuda")
    q_raw, k_raw, v_in = f64(q[0]), f64(k[0]), f64(v[0])
    sk.kv_append(tbl, layer, q, k, v)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = sk.prefill_attention(q, k, v, 0, S, W, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and layer.error_bits() == 0
    # ring state and contents after the long chunk (head = 0, count = W)
    ring = RingCache(S, W)
    ring.append(list(range(T)))
    assert (int(layer.pos[0]), int(layer.head[0]), int(layer.count[0])) == (ring.pos, ring.head, ring.count)
    slots = [0, 1, 3, 4, 5, 2000, W + S - 1]
    for s in slots:
        P = ring.slots[s]
        kr = rope_rotate(k_raw[P:P + 1], [P], spec.omega(), 1.0, D)[0]
        assert_rows_close(f64(layer.k[0, :, s]), kr, torch.bfloat16)
        assert np.array_equal(f64(layer.v[0, :, s]), v_in[P])
    # attention: the oracle rotates the raw Q/K itself
    qr = rope_rotate(q_raw, np.arange(T), spec.omega(), 1.0, D)
    kr = rope_rotate(k_raw, np.arange(T), spec.omega(), 1.0, D)
    assert_rows_close(f64(q[0, :64]), qr[:64], torch.bfloat16)
    rng = np.random.default_rng(66)
    rows = sorted(set([0, 1, 3, 4, 5, 63, 64, 127, 128, 129, 4090, 4091, 4092, 4095, 4096, 4097, 4223, 8191,
                       8192, T - 129, T - 128, T - 1] + rng.integers(0, T, 40).tolist()))
    want = o_prefill(qr, kr, v_in, 0, S, W, rows=rows)
    got = f64(out[0, rows])
    worst = float(np.abs(got - want).max())
    assert worst <= BF16_ATTN_ATOL, worst
