"""GPU parity: turning the recent keys of ring layers by a uniform number of positions
(local-position caches, "Attention Sink 与 Streaming KV Cache", "RoPE：absolute
positions 与 local rerotation 是两种实现"), bf16 and int8 keys, against the float64
oracle."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import (RingCache, dequantize_int8_rows, quantize_int8_rows, rope_inv_freq,
                                  rope_rotate, shift_recent_keys)
from tests.test_gpu_rerotate import assert_int8_requant
from tests.test_gpu_rope_append_decode import assert_rows_close, bf16_ulp, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def _rings(sk, B, Hkv, D, S, W, kdtype, seed, lengths):
    """Two ring layers with random contents and the states the oracle's ring machine
    reaches after `lengths` tokens per sequence (some full and wrapped, some not)."""
    from sink_kv_attention_gb300 import synth
    layers, states = [], []
    for i in range(2):
        L = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=kdtype)
        rcs = []
        for b, n in enumerate(lengths[i]):
            rc = RingCache(S, W)
            rc.append(list(range(n)))
            rcs.append(rc)
        L.pos.copy_(torch.tensor([rc.pos for rc in rcs]))
        L.head.copy_(torch.tensor([rc.head for rc in rcs], dtype=torch.int32))
        L.count.copy_(torch.tensor([rc.count for rc in rcs], dtype=torch.int32))
        if kdtype == torch.bfloat16:
            synth.fill_normal_(L.k, seed + i)
        else:
            L.k.copy_(synth.randint(L.k.shape, seed + i, -127, 128).to(torch.int8))
            L.k_scale.copy_(synth.uniform(L.k_scale.shape, seed + 10 + i, 0.001, 0.02))
        synth.fill_normal_(L.v, seed + 20 + i)
        layers.append(L)
        states.append(rcs)
    return layers, states


@pytest.mark.parametrize("kdt", ["bf16", "i8"])
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("D,r,delta", [(128, 64, -1), (128, 128, -3), (64, 64, 2), (128, 64, -700)])
def test_shift_recent_matches_oracle(sk, kdt, neox, D, r, delta):
    B, Hkv, S, W = 2, 2, 3, 500
    kdtype = torch.bfloat16 if kdt == "bf16" else torch.int8
    table = sk.RopeTable(D, r, 1e4, 1024, neox=neox)
    om = rope_inv_freq(r, 1e4)
    layers, states = _rings(sk, B, Hkv, D, S, W, kdtype, 30, [[2, 1900], [700, 301]])
    k_in = [L.k.clone() for L in layers]
    s_in = [None if L.k_scale is None else L.k_scale.clone() for L in layers]
    v_in = [L.v.clone() for L in layers]
    sk.kv_shift_recent(layers, table, delta)
    torch.cuda.synchronize()
    for i, L in enumerate(layers):
        assert torch.equal(L.v, v_in[i])
        for b in range(B):
            rc = states[i][b]
            recent = [S + j for j in range(rc.count)]
            other = [s for s in range(S + W) if s not in set(recent)]
            got = L.k[b].transpose(0, 1)          # [slot, Hkv, D]
            before = k_in[i][b].transpose(0, 1)
            assert torch.equal(got[other], before[other])   # sinks and empty slots untouched
            if not recent:
                continue
            if kdt == "bf16":
                # the oracle's own shift on a cache holding the same rows
                oc = RingCache(S, W)
                oc.count = rc.count
                oc.slots = [(f64(before[s]), None) if s in set(recent) else None for s in range(S + W)]
                shift_recent_keys(oc, delta, om, r, neox)
                want = np.stack([oc.slots[s][0] for s in recent])
                assert_rows_close(f64(got[recent]), want, torch.bfloat16)
            else:
                sc_in = s_in[i][b].transpose(0, 1)[recent].cpu().numpy()
                x = dequantize_int8_rows(before[recent].cpu().numpy(), sc_in)
                turned = rope_rotate(x, [delta] * len(recent), om, 1.0, r, neox)
                codes_w, scale_w = quantize_int8_rows(turned)
                assert_int8_requant(got[recent].cpu().numpy(), L.k_scale[b].transpose(0, 1)[recent].cpu().numpy(),
                                    codes_w, scale_w, turned)
                sc_other = L.k_scale[b].transpose(0, 1)[other]
                assert torch.equal(sc_other, s_in[i][b].transpose(0, 1)[other])
        assert L.error_bits() == 0


def test_page_example_local_positions_through_the_library(sk):
    """Page 4's C=6, S=2 cache after 10 tokens with keys rotated at their local
    positions (sinks 0, 1; recent 2..5): shifting by -1 gives the keys rotated at local
    1..4 from the raw keys (two bf16 roundings: within 2 ulps of the row max); the
    sink keys stay bit for bit."""
    from sink_kv_attention_gb300 import synth
    D, S, W, T = 128, 2, 4, 10
    table = sk.RopeTable(D, D, 1e4, 64)
    om = rope_inv_freq(D, 1e4)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, 1, D, sinks=S, window=W)
    rc = RingCache(S, W)
    rc.append(list(range(T)))
    layer.pos.fill_(rc.pos)
    layer.head.fill_(rc.head)
    layer.count.fill_(rc.count)
    raw = synth.normal((T, 1, D), 40, torch.bfloat16, device="cuda")
    chrono = rc.chronological_slots()
    assert [rc.slot_pos[s] for s in chrono] == [0, 1, 6, 7, 8, 9]
    for local, s in enumerate(chrono):
        k = raw[rc.slot_pos[s]].clone()[None]             # [1, 1, D]
        sk.rope_apply(table, k, torch.tensor([local], device="cuda"))
        layer.k[0, 0, s] = k[0, 0]
    sinks_before = layer.k[0, 0, :S].clone()
    sk.kv_shift_recent([layer], table, -1)
    torch.cuda.synchronize()
    assert torch.equal(layer.k[0, 0, :S], sinks_before)
    for local, s in enumerate(chrono[S:], start=S):
        want = rope_rotate(f64(raw[rc.slot_pos[s]])[None], [local - 1], om, 1.0, D)[0, 0]
        got = f64(layer.k[0, 0, s])
        assert np.all(np.abs(got - want) <= 2 * bf16_ulp(np.abs(want).max()) + 1e-6)


def test_shift_arguments(sk):
    table = sk.RopeTable(64, 64, 1e4, 16)
    ring = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, 1, 64, sinks=1, window=8)
    glob = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, 1, 64, capacity=8)
    with pytest.raises(sk.SinkKVError) as e:
        sk.kv_shift_recent([glob], table, -1)
    assert e.value.status == sk.SK_ERR_ARG
    with pytest.raises(sk.SinkKVError) as e:
        sk.kv_shift_recent([ring], table, -16)
    assert e.value.status == sk.SK_ERR_POSITION_RANGE
    before = ring.k.clone()
    sk.kv_shift_recent([ring], table, 0)
    assert torch.equal(ring.k, before)
