"""GPU parity: split-K decode attention over int8 K caches (codes + one fp32 scale per
row, bf16 values and queries), against the float64 oracle.  The oracle takes the cache
as given: each key is code * scale in float64."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import GlobalCache, RingCache, RopeSpec, attend, quantize_int8_rows, rope_rotate
from sink_kv_attention_gb300 import synth
from tests.test_gpu_rerotate import assert_int8_requant
from tests.test_gpu_rope_append_decode import f64, BF16_ATTN_ATOL

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def _dequant_keys(layer, b):
    """[Hkv, C, D] float64 keys of sequence b: code * scale."""
    return f64(layer.k[b].to(torch.float32)) * f64(layer.k_scale[b])[..., None]


@pytest.mark.parametrize("kind", ["ring", "global"])
@pytest.mark.parametrize("Dh,r", [(128, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("neox", [True, False])
def test_int8_append_codes_match_oracle_quantisation(sk, kind, Dh, r, neox):
    """The quantising append, code by code: every stored row's codes and scale against
    the oracle's int8 rule on the float64 rotated key, quantize_int8_rows(rope_rotate(k))
    ("#2961 rope: --rope-scaling dynamic", "What it does": int8 K, one scale per row).
    Codes are exact except within 1e-3 of a rounding tie; scales within 1e-5 relative.
    Chunks of one token (decode mode) and longer ones, ring wrap and global prefix;
    rows of zeros get scale 1 and codes 0."""
    B, Hq, Hkv, S, W = 2, 8, 2, 3, 29
    chunks = [1, 4, 1, 17, 2, 40, 1, 9]
    total = sum(chunks)
    tbl = sk.RopeTable(Dh, r, 1e4, 512, neox=neox)
    spec = RopeSpec(Dh, r, 1e4, neox)
    if kind == "ring":
        layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, Dh, sinks=S, window=W, k_dtype=torch.int8)
        caches = [RingCache(S, W) for _ in range(B)]
    else:
        layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, Dh, capacity=total + 5, k_dtype=torch.int8)
        caches = [GlobalCache(total + 5) for _ in range(B)]
    k_all = synth.normal((B, total, Hkv, Dh), 43, torch.bfloat16)
    k_all[1, 5, 0] = 0.0                      # a zero row: scale 1, codes 0
    v_all = synth.normal((B, total, Hkv, Dh), 44, torch.bfloat16)
    want_codes, want_scale, turned = [], [], []
    for b in range(B):
        kr = rope_rotate(f64(k_all[b]), np.arange(total), spec.omega(), 1.0, r, neox)   # [total, Hkv, D]
        c_, s_ = quantize_int8_rows(kr)
        want_codes.append(c_)
        want_scale.append(s_)
        turned.append(kr)
    done = 0
    for T in chunks:
        sk.kv_append(tbl, layer, None, k_all[:, done:done + T].clone().cuda(), v_all[:, done:done + T].clone().cuda())
        for b in range(B):
            caches[b].append([done + t for t in range(T)])
        done += T
        torch.cuda.synchronize()
        codes, scales = layer.k.cpu().numpy(), layer.k_scale.cpu().numpy()
        for b in range(B):
            if kind == "ring":
                slots = caches[b].chronological_slots()
                held = caches[b].chronological_positions()
            else:
                slots = held = list(range(done))
            got_c = codes[b][:, slots].transpose(1, 0, 2)          # [n, Hkv, D]
            got_s = scales[b][:, slots].transpose(1, 0)            # [n, Hkv]
            assert_int8_requant(got_c, got_s, want_codes[b][held], want_scale[b][held], turned[b][held])
            assert np.array_equal(f64(layer.v[b][:, slots].transpose(0, 1)), f64(v_all[b, held]))
    assert want_scale[1][5, 0] == 1.0 and not want_codes[1][5, 0].any()
    if kind == "global":
        assert float(layer.k_scale[1, 0, 5]) == 1.0 and not layer.k[1, 0, 5].any()
    assert layer.error_bits() == 0


@pytest.mark.parametrize("kind", ["ring", "global"])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 4), (4, 4), (8, 4)])
def test_int8_key_decode_through_appends(sk, kind, Hq, Hkv):
    """Chunks appended through the library (RoPE, quantise K per row), then the last
    query of each chunk decoded over the int8 cache: the rows the oracle's cache holds
    at each step, with the keys the device stored."""
    B, S, W = 2, 3, 37
    chunks = [1, 5, 17, 2, 40, 1, 9, 1]
    total = sum(chunks)
    tbl = sk.RopeTable(D, D, 1e4, 512)
    spec = RopeSpec(D, D, 1e4)
    if kind == "ring":
        layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=torch.int8)
        caches = [RingCache(S, W) for _ in range(B)]
    else:
        layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, D, capacity=total + 5, k_dtype=torch.int8)
        caches = [GlobalCache(total + 5) for _ in range(B)]
    q_all = synth.normal((B, total, Hq, D), 40, torch.bfloat16)
    k_all = synth.normal((B, total, Hkv, D), 41, torch.bfloat16)
    v_all = synth.normal((B, total, Hkv, D), 42, torch.bfloat16)
    done = 0
    for T in chunks:
        q = q_all[:, done:done + T].clone().cuda()
        sk.kv_append(tbl, layer, q, k_all[:, done:done + T].clone().cuda(), v_all[:, done:done + T].clone().cuda())
        for b in range(B):
            # the oracle's cache records positions; its rows are read back from the device
            caches[b].append([done + t for t in range(T)])
        done += T
        out = f64(sk.decode_attention(layer, q[:, -1].contiguous()))
        torch.cuda.synchronize()
        for b in range(B):
            keys = _dequant_keys(layer, b)
            vals = f64(layer.v[b])
            if kind == "ring":
                slots = caches[b].chronological_slots()
            else:
                slots = list(range(done))
            qr = rope_rotate(f64(q_all[b, done - 1:done]), [done - 1], spec.omega(), 1.0, D)[0]
            want = attend(qr, keys[:, slots].transpose(1, 0, 2), vals[:, slots].transpose(1, 0, 2))
            np.testing.assert_allclose(out[b], want, rtol=0, atol=BF16_ATTN_ATOL)
        if kind == "ring":
            assert layer.head.tolist() == [c.head for c in caches]
            assert layer.count.tolist() == [c.count for c in caches]
    assert layer.error_bits() == 0


def test_int8_key_decode_matches_bf16_decode_of_the_same_keys(sk):
    """The int8 path against the library's bf16 path on the dequantised keys (rounded to
    bf16) and the oracle: the three agree within the bf16 attention tolerance."""
    B, Hq, Hkv, S, W = 4, 16, 4, 4, 300
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=torch.int8)
    layer.k.copy_(synth.randint(layer.k.shape, 43, -127, 128, device="cuda").to(torch.int8))
    synth.fill_uniform_(layer.k_scale, 44, 0.5 / 127, 2.0 / 127)
    synth.fill_normal_(layer.v, 45)
    pos, head, count = synth.window_state(46, B, W, 200, 5000)
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    q = synth.normal((B, Hq, D), 47, torch.bfloat16, device="cuda")
    out8 = f64(sk.decode_attention(layer, q))
    ref = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    ref.k.copy_((layer.k.to(torch.float32) * layer.k_scale[..., None]).to(torch.bfloat16))
    ref.v.copy_(layer.v)
    ref.pos.copy_(layer.pos)
    ref.head.copy_(layer.head)
    ref.count.copy_(layer.count)
    out16 = f64(sk.decode_attention(ref, q))
    torch.cuda.synchronize()
    for b in range(B):
        n = min(int(pos[b]), S) + int(count[b])
        keys = _dequant_keys(layer, b)[:, :n].transpose(1, 0, 2)
        vals = f64(layer.v[b])[:, :n].transpose(1, 0, 2)
        want = attend(f64(q[b]), keys, vals)
        np.testing.assert_allclose(out8[b], want, rtol=0, atol=BF16_ATTN_ATOL)
        np.testing.assert_allclose(out16[b], want, rtol=0, atol=BF16_ATTN_ATOL)


def test_int8_key_decode_learned_sinks_noalloc_and_full_size(sk):
    """The windowed decode shapes (B=32, H_q=32, H_kv=8, S=4, W=4092) on an int8 K
    cache, with learned sinks, through the no-alloc call; sampled sequences."""
    c = synth.WINDOW
    B, Hq, Hkv, S, W = c["B"], c["Hq"], c["Hkv"], c["S"], c["W"]
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=torch.int8)
    layer.k.copy_(synth.randint(layer.k.shape, 48, -127, 128, device="cuda").to(torch.int8))
    synth.fill_uniform_(layer.k_scale, 49, 0.5 / 127, 2.0 / 127)
    synth.fill_normal_(layer.v, 50)
    pos, head, count = synth.window_state(51, B, W, c["pos_lo"], c["pos_hi"])
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    q = synth.normal((B, Hq, D), 52, torch.bfloat16, device="cuda")
    z = torch.linspace(-12.0, 16.0, Hq)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    out = f64(sk.decode_attention_noalloc(layer, q, out, sink_logits=z.cuda()))
    torch.cuda.synchronize()
    for b in (0, 7, 19, 31):
        n = min(int(pos[b]), S) + int(count[b])
        keys = _dequant_keys(layer, b)[:, :n].transpose(1, 0, 2)
        vals = f64(layer.v[b])[:, :n].transpose(1, 0, 2)
        want = attend(f64(q[b]), keys, vals, sink_logits=z.numpy())
        np.testing.assert_allclose(out[b], want, rtol=0, atol=BF16_ATTN_ATOL)
    assert layer.error_bits() == 0
