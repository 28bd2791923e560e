"""GPU parity: in-place rerotation of cached keys on a RoPE factor change, bf16 and
int8 + per-row scale, against the float64 oracle."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import (RingCache, RopeSpec, dequantize_int8_rows, quantize_int8_rows, rerotate,
                                  rerotate_int8, rope_rotate)
from tests.test_gpu_rope_append_decode import assert_rows_close, bf16_ulp, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def assert_int8_requant(codes_gpu, scale_gpu, codes_want, scale_want, turned):
    """Scales within 1e-5 relative; codes equal except where the float64 value sits
    within 1e-3 of a rounding tie, where either neighbour is a correct rounding."""
    scale_gpu = np.asarray(scale_gpu, dtype=np.float64)
    scale_want = np.asarray(scale_want, dtype=np.float64)
    np.testing.assert_allclose(scale_gpu, scale_want, rtol=1e-5)
    q = turned / scale_want[..., None]
    near_tie = np.abs(np.abs(q - np.trunc(q)) - 0.5) < 1e-3
    diff = np.abs(codes_gpu.astype(np.int32) - codes_want.astype(np.int32))
    assert np.all(diff[~near_tie] == 0), int(diff[~near_tie].max())
    assert np.all(diff <= 1)


def _specs(D, r, neox, L0, fa, fb):
    a = RopeSpec(D, r, 5e5, neox, fa, L0)
    return a, a.with_factor(fb)


@pytest.mark.parametrize("kdt", ["bf16", "i8"])
@pytest.mark.parametrize("neox", [True, False])
def test_rerotate_all_rows_ring_and_global(sk, kdt, neox):
    from sink_kv_attention_gb300 import synth
    D, r, Hkv, B, L0 = 128, 64, 2, 2, 2048
    S, W = 3, 700
    fa, fb = 1.0, 2.0
    tA = sk.RopeTable(D, r, 5e5, 8192, neox=neox, yarn_factor=fa, yarn_orig_ctx=L0)
    tB = sk.RopeTable(D, r, 5e5, 8192, neox=neox, yarn_factor=fb, yarn_orig_ctx=L0)
    specA, specB = _specs(D, r, neox, L0, fa, fb)
    kdtype = torch.bfloat16 if kdt == "bf16" else torch.int8
    glob = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, D, capacity=6000, k_dtype=kdtype)
    ring = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=kdtype)
    glob.pos.copy_(torch.tensor([5000, 3333]))
    # ring states from the oracle's own state machine (token-by-token appends)
    rings = []
    for b, n in enumerate([5000, 200]):
        rc = RingCache(S, W)
        for p in range(n):
            rc.append([p])
        rings.append(rc)
    ring.pos.copy_(torch.tensor([rc.pos for rc in rings]))
    ring.head.copy_(torch.tensor([rc.head for rc in rings], dtype=torch.int32))
    ring.count.copy_(torch.tensor([rc.count for rc in rings], dtype=torch.int32))
    for i, L in enumerate([glob, ring]):
        if kdt == "bf16":
            synth.fill_normal_(L.k, 50 + i)
        else:
            L.k.copy_(synth.randint(L.k.shape, 52 + i, -127, 128).to(torch.int8))
            L.k_scale.copy_(synth.uniform(L.k_scale.shape, 54 + i, 0.001, 0.02))
    k_in = [L.k.clone() for L in (glob, ring)]
    s_in = [None if L.k_scale is None else L.k_scale.clone() for L in (glob, ring)]
    sk.kv_rerotate([glob, ring], tA, tB)
    torch.cuda.synchronize()
    for i, L in enumerate([glob, ring]):
        for b in range(B):
            if L is glob:
                slots = list(range(int(glob.pos[b])))
                positions = slots
            else:
                slots = [s for s in range(S + W) if rings[b].slot_pos[s] >= 0]
                positions = [rings[b].slot_pos[s] for s in slots]
            empty = [s for s in range(L.capacity) if s not in set(slots)]
            got = L.k[b].transpose(0, 1)    # [slot, Hkv, D]
            before = k_in[i][b].transpose(0, 1)
            assert torch.equal(got[empty], before[empty])   # empty slots untouched
            if kdt == "bf16":
                want = rerotate(f64(before[slots]), positions, specA, specB)
                assert_rows_close(f64(got[slots]), want, torch.bfloat16)
            else:
                sc_in = s_in[i][b].transpose(0, 1)[slots].cpu().numpy()
                codes_w, scale_w, turned = rerotate_int8(before[slots].cpu().numpy(), sc_in, positions, specA, specB)
                assert_int8_requant(got[slots].cpu().numpy(), L.k_scale[b].transpose(0, 1)[slots].cpu().numpy(),
                                    codes_w, scale_w, turned)
        assert L.error_bits() == 0


@pytest.mark.parametrize("kdt", ["bf16", "i8"])
def test_rerotate_full_size_sampled(sk, kdt):
    """48 layers x 4 kv heads x 524288 cached positions, r = 64 of d_h = 128, YaRN
    L0 = 262144, factor 1 -> 2; 4096 sampled rows checked against the oracle."""
    from sink_kv_attention_gb300 import synth
    c = synth.REROTATE
    D, r, Hkv, N, nl = c["D"], c["r"], c["Hkv"], c["positions"], c["layers"]
    tA = sk.RopeTable(D, r, c["theta"], N, yarn_factor=c["factor_a"], yarn_orig_ctx=c["orig_ctx"])
    tB = sk.RopeTable(D, r, c["theta"], N, yarn_factor=c["factor_b"], yarn_orig_ctx=c["orig_ctx"])
    specA = RopeSpec(D, r, c["theta"], True, c["factor_a"], c["orig_ctx"])
    specB = specA.with_factor(c["factor_b"])
    kdtype = torch.bfloat16 if kdt == "bf16" else torch.int8
    layers = []
    for l in range(nl):
        L = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, Hkv, D, capacity=N, k_dtype=kdtype, with_v=False)
        L.pos.fill_(N)
        if kdt == "bf16":
            synth.fill_uniform_(L.k, 500 + l, -1.0, 1.0)
        else:
            L.k.copy_(synth.randint(L.k.shape, 600 + l, -127, 128, device="cuda").to(torch.int8))
            synth.fill_uniform_(L.k_scale, 700 + l, 1.0 / 127, 2.0 / 127)
        layers.append(L)
    idx_l = synth.randint((4096,), 9, 0, nl)
    idx_g = synth.randint((4096,), 10, 0, Hkv)
    idx_s = synth.randint((4096,), 11, 0, N)
    idx_s[:4] = torch.tensor([0, 1, N - 1, 262144])
    before = torch.stack([layers[l].k[0, g, s] for l, g, s in zip(idx_l.tolist(), idx_g.tolist(), idx_s.tolist())])
    sc_before = (torch.stack([layers[l].k_scale[0, g, s] for l, g, s in zip(idx_l.tolist(), idx_g.tolist(), idx_s.tolist())])
                 if kdt == "i8" else None)
    sk.kv_rerotate(layers, tA, tB)
    torch.cuda.synchronize()
    after = torch.stack([layers[l].k[0, g, s] for l, g, s in zip(idx_l.tolist(), idx_g.tolist(), idx_s.tolist())])
    pos = idx_s.numpy()
    if kdt == "bf16":
        want = rerotate(f64(before)[:, None, :], pos, specA, specB)[:, 0]
        assert_rows_close(f64(after), want, torch.bfloat16)
    else:
        sc_after = torch.stack([layers[l].k_scale[0, g, s] for l, g, s in zip(idx_l.tolist(), idx_g.tolist(), idx_s.tolist())])
        codes_w, scale_w, turned = rerotate_int8(before.cpu().numpy()[:, None, :], sc_before.cpu().numpy()[:, None],
                                                 pos, specA, specB)
        assert_int8_requant(after.cpu().numpy(), sc_after.cpu().numpy(), codes_w[:, 0], scale_w[:, 0], turned[:, 0])
    assert all(L.error_bits() == 0 for L in layers)


@pytest.mark.parametrize("kdt", ["bf16", "i8"])
def test_turned_vs_written_at_new_factor(sk, kdt):
    """Page 3's yardstick: keys written at factor A by the append kernel and turned to
    B, against keys written directly at B, both measured from the float64 key at B:
    RMS ratio <= 1.6x; worst element <= 3 bf16 ulps of the row max, or <= 2 int8 steps."""
    from sink_kv_attention_gb300 import synth
    D, r, Hkv, N, L0 = 128, 64, 4, 524288, 262144
    tA = sk.RopeTable(D, r, 5e5, N, yarn_factor=1.0, yarn_orig_ctx=L0)
    tB = sk.RopeTable(D, r, 5e5, N, yarn_factor=2.0, yarn_orig_ctx=L0)
    specA, specB = _specs(D, r, True, L0, 1.0, 2.0)
    kdtype = torch.bfloat16 if kdt == "bf16" else torch.int8
    raw = synth.uniform((1, N, Hkv, D), 77, -1.0, 1.0, torch.bfloat16, device="cuda")
    v = torch.zeros_like(raw)
    la = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, Hkv, D, capacity=N, k_dtype=kdtype)
    lb = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, Hkv, D, capacity=N, k_dtype=kdtype)
    sk.kv_append(tA, la, None, raw.clone(), v)
    sk.kv_append(tB, lb, None, raw.clone(), v)
    sk.kv_rerotate([la], tA, tB)
    torch.cuda.synchronize()
    rows = synth.randint((8192,), 78, 0, N)
    g = synth.randint((8192,), 79, 0, Hkv)
    exact = rope_rotate(f64(raw[0, rows, g])[:, None, :], rows.numpy(), specB.omega(), specB.mscale(), r)[:, 0]

    def read(L):
        k = L.k[0, g, rows]
        if kdt == "bf16":
            return f64(k), None
        sc = L.k_scale[0, g, rows]
        return dequantize_int8_rows(k.cpu().numpy(), sc.cpu().numpy()), sc.cpu().numpy()

    turned, _ = read(la)
    written, sc_b = read(lb)
    rms_t = np.sqrt(np.mean((turned - exact) ** 2))
    rms_w = np.sqrt(np.mean((written - exact) ** 2))
    assert rms_t / rms_w <= 1.6
    if kdt == "bf16":
        ulp_rowmax = bf16_ulp(np.abs(exact).max(axis=-1, keepdims=True))
        assert np.max(np.abs(turned - exact) / ulp_rowmax) <= 3.0
    else:
        assert np.max(np.abs(turned - exact) / sc_b[:, None]) <= 2.0
    assert la.error_bits() == 0 and lb.error_bits() == 0
