"""GPU parity: RoPE apply, fused RoPE + append (ring with sinks, global prefix) and
split-K decode attention, through the C ABI, against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import (GlobalCache, RingCache, RopeSpec, decode_attention as o_decode,
                                  rope_rotate)
from tests.conftest import golden_path

pytestmark = pytest.mark.gpu

BF16_ATTN_ATOL = 2e-2   # bf16 attention outputs, N(0,1) inputs
F32_ATTN_ATOL = 2e-5    # fp32 attention outputs (fp32 accumulation, exp2 of base-2 logits)


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def f64(t):
    return t.detach().float().cpu().double().numpy()


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 1e-30)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def assert_rows_close(got, want, dtype):
    """fp32: per-row max error <= 1e-5 of the row max; bf16: 1 ulp + 1e-5 of the row max."""
    rowmax = np.abs(want).max(axis=-1, keepdims=True)
    err = np.abs(got - want)
    if dtype == torch.float32:
        assert np.all(err <= 1e-5 * rowmax + 1e-30), float((err / (rowmax + 1e-30)).max())
    else:
        assert np.all(err <= bf16_ulp(want) + 1e-5 * rowmax), float((err - bf16_ulp(want)).max())


# ---------------------------------------------------------------------------
# RoPE apply
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D,r", [(64, 64), (128, 128), (128, 64)])
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("factor", [1.0, 2.0])
def test_rope_apply_matches_oracle(sk, dtype, D, r, neox, factor):
    from sink_kv_attention_gb300 import synth
    max_pos = 600000
    table = sk.RopeTable(D, r, 5e5, max_pos, neox=neox, yarn_factor=factor, yarn_orig_ctx=262144)
    n_tok, H = 777, 3
    x = synth.normal((n_tok, H, D), seed=5, dtype=dtype).cuda()
    pos = synth.randint((n_tok,), seed=6, lo=0, hi=max_pos)
    pos[:4] = torch.tensor([0, 1, max_pos - 1, 524287])
    x_in = f64(x)
    sk.rope_apply(table, x, pos.cuda())
    spec = RopeSpec(D, r, 5e5, neox, factor, 262144)
    want = rope_rotate(x_in, pos.numpy(), spec.omega(), spec.mscale(), r, neox)
    assert_rows_close(f64(x), want, dtype)
    if r < D:
        assert torch.equal(torch.from_numpy(f64(x)[..., r:]), torch.from_numpy(x_in[..., r:]))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("H", [17, 40])
def test_rope_apply_many_heads(sk, dtype, D, neox, H):
    """Tokens of many heads: the kernel takes a token's rows in passes of several row
    groups, so these head counts need more than one pass and end on a partial one."""
    from sink_kv_attention_gb300 import synth
    max_pos = 70000
    table = sk.RopeTable(D, D, 1e4, max_pos, neox=neox)
    n_tok = 301
    x = synth.normal((n_tok, H, D), seed=7, dtype=dtype).cuda()
    pos = synth.randint((n_tok,), seed=8, lo=0, hi=max_pos)
    x_in = f64(x)
    sk.rope_apply(table, x, pos.cuda())
    spec = RopeSpec(D, D, 1e4, neox)
    want = rope_rotate(x_in, pos.numpy(), spec.omega(), spec.mscale(), D, neox)
    assert_rows_close(f64(x), want, dtype)


def test_rope_apply_full_chunk_sampled(sk):
    """The Q of a 32,768-token chunk at positions 32768.. (H_q=32, d_h=r=128, theta 5e5),
    as a chunk prefilled over a cached prefix rotates it; sampled tokens."""
    from sink_kv_attention_gb300 import synth
    T, H, D, p0 = 32768, 32, 128, 32768
    table = sk.RopeTable(D, D, 5e5, p0 + T)
    x = synth.normal((T, H, D), seed=9, dtype=torch.bfloat16, device="cuda")
    x_in = x.cpu()
    sk.rope_apply(table, x, torch.arange(p0, p0 + T, dtype=torch.int64, device="cuda"))
    rows = [0, 1, 7, 8, 4095, 16384, T - 2, T - 1]
    spec = RopeSpec(D, D, 5e5, True)
    want = rope_rotate(f64(x_in[rows]), [p0 + t for t in rows], spec.omega(), spec.mscale(), D, True)
    assert_rows_close(f64(x[rows]), want, torch.bfloat16)


def test_rope_apply_position_out_of_range_is_flagged(sk):
    table = sk.RopeTable(64, 64, 1e4, 100)
    x = torch.randn(3, 2, 64, device="cuda")
    before = x.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sk.rope_apply(table, x, torch.tensor([5, 100, -1], device="cuda"), err=err)
    assert int(err.item()) & sk.SK_DEVERR_POSITION_RANGE
    assert torch.equal(x[1:], before[1:])       # rows 1 and 2 untouched
    assert not torch.equal(x[0], before[0])     # row 0 rotated


# ---------------------------------------------------------------------------
# The tiny workload: the page's C=6, S=2, T=10 visible table, fp32
# ---------------------------------------------------------------------------

def _golden_table():
    rows = {}
    with open(golden_path("visible_c6_s2_t10.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            i, vis = line.split(":")
            rows[int(i)] = [int(x) for x in vis.split(",")]
    return rows


def test_tiny_decode_reproduces_visible_table(sk):
    from sink_kv_attention_gb300 import synth
    c = synth.TINY
    table_rows = _golden_table()
    tbl = sk.RopeTable(c["D"], c["r"], c["theta"], 64)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, c["Hkv"], c["D"], sinks=c["S"], window=c["W"],
                                k_dtype=torch.float32, v_dtype=torch.float32)
    q_all = synth.normal((1, c["T"], c["Hq"], c["D"]), seed=0)
    k_all = synth.normal((1, c["T"], c["Hkv"], c["D"]), seed=1)
    v_all = synth.normal((1, c["T"], c["Hkv"], c["D"]), seed=2)
    spec = RopeSpec(c["D"], c["r"], c["theta"])
    ring = RingCache(c["S"], c["W"])
    for t in range(c["T"]):
        q = q_all[:, t:t + 1].clone().cuda()
        k = k_all[:, t:t + 1].clone().cuda()
        v = v_all[:, t:t + 1].clone().cuda()
        sk.kv_append(tbl, layer, q, k, v)
        out = sk.decode_attention(layer, q[:, 0].contiguous())
        qr = rope_rotate(f64(q_all[0, t:t + 1]), [t], spec.omega(), 1.0, c["r"])
        kr = rope_rotate(f64(k_all[0, t:t + 1]), [t], spec.omega(), 1.0, c["r"])
        ring.append([(kr[0], f64(v_all[0, t]))])
        assert_rows_close(f64(q[0]), qr, torch.float32)
        assert (int(layer.pos[0]), int(layer.head[0]), int(layer.count[0])) == (ring.pos, ring.head, ring.count)
        # which positions the cache holds: V rows are copied exactly, so match them
        occupied = min(ring.pos, c["S"]) + int(layer.count[0])
        held = []
        v_gpu = f64(layer.v[0, 0])
        for s in range(occupied):
            match = [p for p in range(t + 1) if np.array_equal(v_gpu[s], f64(v_all[0, p, 0]))]
            assert len(match) == 1
            held.append(match[0])
        assert sorted(held) == table_rows[t]
        np.testing.assert_allclose(f64(out[0]), o_decode(ring, qr[0]), rtol=0, atol=F32_ATTN_ATOL)


def test_decode_visible_set_probe(sk):
    """q = 0 makes the softmax uniform, so out = mean of the visible V rows: with V
    one-hot per position, out > 0 exactly on the visible positions."""
    S, W, T, D = 2, 4, 14, 64
    tbl = sk.RopeTable(D, D, 1e4, 64)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, 1, D, sinks=S, window=W,
                                k_dtype=torch.float32, v_dtype=torch.float32)
    for t in range(T):
        q = torch.zeros(1, 1, 1, D, device="cuda")
        k = torch.randn(1, 1, 1, D, device="cuda")
        v = torch.zeros(1, 1, 1, D, device="cuda")
        v[0, 0, 0, t] = 1.0
        sk.kv_append(tbl, layer, q, k, v)
        out = sk.decode_attention(layer, q[:, 0].contiguous())[0, 0].cpu().numpy()
        from oracle.sinkkv_oracle import visible_positions
        vis = visible_positions(t, S + W, S)
        assert [i for i in range(D) if out[i] > 0] == vis
        np.testing.assert_allclose(out[vis], 1.0 / len(vis), rtol=1e-6)


# ---------------------------------------------------------------------------
# Chunked appends: the ring state machine and the global prefix
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("kind", ["ring", "global"])
@pytest.mark.parametrize("D,r", [(128, 64), (64, 64), (128, 128)])
@pytest.mark.parametrize("neox", [True, False])
def test_chunked_append_state_and_decode(sk, dtype, kind, D, r, neox):
    """Fused RoPE + append, chunk by chunk, in NeoX (j, j + r/2) and GPT-J (2j, 2j + 1)
    pairing ("RoPE, scaling, sliding window, attention sinks", RoPE section: the two
    pairings give different keys), partial rotary included: rotated Q and K, cached
    rows and ring state against the oracle, then a decode over the cache."""
    from sink_kv_attention_gb300 import synth
    B, Hq, Hkv, S, W = 2, 8, 2, 3, 5
    chunks = [1, 2, 3, 5, 7, 1, 11, 4, 1, 6, 1, 1]
    total = sum(chunks)
    tbl = sk.RopeTable(D, r, 1e4, 256, neox=neox)
    spec = RopeSpec(D, r, 1e4, neox)
    if kind == "ring":
        layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=dtype, v_dtype=dtype)
        caches = [RingCache(S, W) for _ in range(B)]
    else:
        layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, D, capacity=total + 3, k_dtype=dtype, v_dtype=dtype)
        caches = [GlobalCache(total + 3) for _ in range(B)]
    q_all = synth.normal((B, total, Hq, D), seed=20, dtype=dtype)
    k_all = synth.normal((B, total, Hkv, D), seed=21, dtype=dtype)
    v_all = synth.normal((B, total, Hkv, D), seed=22, dtype=dtype)
    done = 0
    for T in chunks:
        q = q_all[:, done:done + T].clone().cuda()
        k = k_all[:, done:done + T].clone().cuda()
        v = v_all[:, done:done + T].clone().cuda()
        sk.kv_append(tbl, layer, q, k, v)
        pos = list(range(done, done + T))
        for b in range(B):
            qr = rope_rotate(f64(q_all[b, done:done + T]), pos, spec.omega(), 1.0, r, neox)
            kr = rope_rotate(f64(k_all[b, done:done + T]), pos, spec.omega(), 1.0, r, neox)
            assert_rows_close(f64(q[b]), qr, dtype)
            assert_rows_close(f64(k[b]), kr, dtype)
            caches[b].append([(kr[t], f64(v_all[b, done + t])) for t in range(T)])
        done += T
        assert layer.pos.tolist() == [c.pos for c in caches]
        if kind == "ring":
            assert layer.head.tolist() == [c.head for c in caches]
            assert layer.count.tolist() == [c.count for c in caches]
            for b in range(B):
                for s in range(S + W):
                    if caches[b].slots[s] is None:
                        continue
                    kr_s, v_s = caches[b].slots[s]
                    assert np.array_equal(f64(layer.v[b, :, s]), v_s)
                    assert_rows_close(f64(layer.k[b, :, s]), kr_s, dtype)
        # decode attention of the chunk's last query over the cache
        out = sk.decode_attention(layer, q[:, -1].contiguous())
        for b in range(B):
            qr_last = rope_rotate(f64(q_all[b, done - 1:done]), [done - 1], spec.omega(), 1.0, r, neox)[0]
            want = o_decode(caches[b], qr_last)
            tol = F32_ATTN_ATOL if dtype == torch.float32 else BF16_ATTN_ATOL
            np.testing.assert_allclose(f64(out[b]), want, rtol=0, atol=tol)
    assert layer.error_bits() == 0


def test_global_capacity_overflow_is_flagged(sk):
    D = 64
    tbl = sk.RopeTable(D, D, 1e4, 64)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, 1, D, capacity=8, k_dtype=torch.float32,
                                v_dtype=torch.float32)
    mk = lambda T: torch.randn(1, T, 1, D, device="cuda")
    sk.kv_append(tbl, layer, None, mk(6), mk(6))
    before = layer.k.clone()
    sk.kv_append(tbl, layer, None, mk(3), mk(3))
    assert layer.error_bits() & sk.SK_DEVERR_CAPACITY
    assert int(layer.pos[0]) == 6 and torch.equal(layer.k, before)


def test_sync_check_reports_and_clears_device_errors(sk):
    """sk_sync_check: no bits -> SK_OK; a global overflow -> SK_ERR_CAPACITY with the
    bit, cleared on request; a position past the table -> SK_ERR_POSITION_RANGE."""
    D = 64
    tbl = sk.RopeTable(D, D, 1e4, 8)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, 1, D, capacity=4, k_dtype=torch.float32,
                                v_dtype=torch.float32)
    mk = lambda T: torch.randn(1, T, 1, D, device="cuda")
    sk.kv_append(tbl, layer, None, mk(3), mk(3))
    assert sk.sync_check(layer.err) == (sk.SK_OK, 0)
    sk.kv_append(tbl, layer, None, mk(2), mk(2))           # 3 + 2 > 4
    assert sk.sync_check(layer.err, clear=True) == (sk.SK_ERR_CAPACITY, sk.SK_DEVERR_CAPACITY)
    assert sk.sync_check(layer.err) == (sk.SK_OK, 0)
    ring = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, 1, D, sinks=1, window=20, k_dtype=torch.float32,
                               v_dtype=torch.float32)
    sk.kv_append(tbl, ring, None, mk(9), mk(9))           # positions 0..8, table holds 8
    st, bits = sk.sync_check(ring.err)
    assert st == sk.SK_ERR_POSITION_RANGE and bits & sk.SK_DEVERR_POSITION_RANGE


def test_append_position_past_table_is_flagged(sk):
    D = 64
    tbl = sk.RopeTable(D, D, 1e4, 4)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, 1, D, sinks=1, window=7, k_dtype=torch.float32,
                                v_dtype=torch.float32)
    mk = lambda T: torch.randn(1, T, 1, D, device="cuda")
    sk.kv_append(tbl, layer, None, mk(3), mk(3))
    sk.kv_append(tbl, layer, None, mk(2), mk(2))   # positions 3, 4: 4 is past the table
    assert layer.error_bits() & sk.SK_DEVERR_POSITION_RANGE
    assert int(layer.pos[0]) == 3


# ---------------------------------------------------------------------------
# Full-size workloads, sampled against the oracle
# ---------------------------------------------------------------------------

def _ring_from_inputs(S, W, pos, head, count, k_b, v_b):
    """Oracle ring cache holding the given (input) contents and state."""
    ring = RingCache(S, W)
    ring.pos, ring.head, ring.count = int(pos), int(head), int(count)
    for s in range(S + W):
        ring.slots[s] = (k_b[:, s], v_b[:, s])
    return ring


def test_window_decode_step_full_size(sk):
    """The windowed-layer decode step: B=32, H_q=32, H_kv=8, d_h=128, S=4, W=4092,
    positions U[4096, 32768] with a random ring head; RoPE + append + attention."""
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    tbl = sk.RopeTable(D, c["r"], c["theta"], c["pos_hi"] + 2)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 11)
    synth.fill_normal_(layer.v, 12)
    pos, head, count = synth.window_state(13, B, W, c["pos_lo"], c["pos_hi"])
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    k_in, v_in = layer.k.clone(), layer.v.clone()
    q = synth.normal((B, 1, Hq, D), 14, torch.bfloat16).cuda()
    k = synth.normal((B, 1, Hkv, D), 15, torch.bfloat16).cuda()
    v = synth.normal((B, 1, Hkv, D), 16, torch.bfloat16).cuda()
    q_raw, k_raw, v_raw = f64(q), f64(k), f64(v)
    sk.kv_append(tbl, layer, q, k, v)
    out = f64(sk.decode_attention(layer, q[:, 0].contiguous()))
    spec = RopeSpec(D, c["r"], c["theta"])
    worst = 0.0
    for b in range(B):
        P = int(pos[b])
        ring = _ring_from_inputs(S, W, P, head[b], count[b], f64(k_in[b]), f64(v_in[b]))
        qr = rope_rotate(q_raw[b], [P], spec.omega(), 1.0, D)
        kr = rope_rotate(k_raw[b], [P], spec.omega(), 1.0, D)
        ring.append([(kr[0], v_raw[b, 0])])
        assert (int(layer.pos[b]), int(layer.head[b]), int(layer.count[b])) == (ring.pos, ring.head, ring.count)
        slot = S + (int(head[b])) % W
        assert_rows_close(f64(layer.k[b, :, slot]), kr[0], torch.bfloat16)
        assert np.array_equal(f64(layer.v[b, :, slot]), v_raw[b, 0])
        want = o_decode(ring, qr[0])
        worst = max(worst, float(np.abs(out[b] - want).max()))
    assert worst <= BF16_ATTN_ATOL, worst
    assert layer.error_bits() == 0


def test_hybrid_layers_full_size_sampled(sk):
    """One global layer (131072-token prefix) and one sliding layer (S=4, W=4096) of
    the Llama-3-8B-shaped hybrid decode, at full size; sampled sequences checked."""
    from sink_kv_attention_gb300 import synth
    c = synth.HYBRID
    B, Hq, Hkv, D, S, W, prefix = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"], c["prefix"]
    tbl = sk.RopeTable(D, c["r"], c["theta"], prefix + 2)
    spec = RopeSpec(D, c["r"], c["theta"])
    glob = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, D, capacity=prefix + 1)
    slid = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    for i, L in enumerate([glob, slid]):
        synth.fill_normal_(L.k, 30 + 2 * i)
        synth.fill_normal_(L.v, 31 + 2 * i)
        L.pos.fill_(prefix)
    slid.count.fill_(W)
    slid.head.copy_(synth.randint((B,), 34, 0, W).to(torch.int32))
    sample = [0, 9, 15]
    k_in = {id(L): L.k[sample].clone() for L in (glob, slid)}
    v_in = {id(L): L.v[sample].clone() for L in (glob, slid)}
    head_in = slid.head.clone().cpu()
    for i, L in enumerate([glob, slid]):
        q = synth.normal((B, 1, Hq, D), 40 + 3 * i, torch.bfloat16).cuda()
        k = synth.normal((B, 1, Hkv, D), 41 + 3 * i, torch.bfloat16).cuda()
        v = synth.normal((B, 1, Hkv, D), 42 + 3 * i, torch.bfloat16).cuda()
        q_raw, k_raw, v_raw = f64(q), f64(k), f64(v)
        sk.kv_append(tbl, L, q, k, v)
        out = f64(sk.decode_attention(L, q[:, 0].contiguous()))
        assert L.pos.tolist() == [prefix + 1] * B
        for j, b in enumerate(sample):
            qr = rope_rotate(q_raw[b], [prefix], spec.omega(), 1.0, D)
            kr = rope_rotate(k_raw[b], [prefix], spec.omega(), 1.0, D)
            kb, vb = f64(k_in[id(L)][j]), f64(v_in[id(L)][j])
            if L is glob:
                cache = GlobalCache(prefix + 1)
                cache.rows = [(kb[:, s], vb[:, s]) for s in range(prefix)]
            else:
                cache = _ring_from_inputs(S, W, prefix, head_in[b], W, kb, vb)
            cache.append([(kr[0], v_raw[b, 0])])
            want = o_decode(cache, qr[0])
            assert float(np.abs(out[b] - want).max()) <= BF16_ATTN_ATOL
        assert L.error_bits() == 0


def test_decode_maximum_batch(sk):
    """The largest batch the decode kernels take (1024 sequences; the unit prefix scan
    runs 32 rounds), ragged lengths incl. empty rings; sampled sequences against the
    oracle, and 1025 sequences rejected on the host."""
    from sink_kv_attention_gb300 import synth
    B, Hq, Hkv, D, S, W = 1024, 4, 1, 64, 2, 30
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 91)
    synth.fill_normal_(layer.v, 92)
    lens = synth.randint((B,), 93, 0, 60)
    rings = []
    for b in range(B):
        rc = RingCache(S, W)
        rc.append(list(range(int(lens[b]))))
        rings.append(rc)
    layer.pos.copy_(torch.tensor([rc.pos for rc in rings]))
    layer.head.copy_(torch.tensor([rc.head for rc in rings], dtype=torch.int32))
    layer.count.copy_(torch.tensor([rc.count for rc in rings], dtype=torch.int32))
    q = synth.normal((B, Hq, D), 94, torch.bfloat16).cuda()
    out = f64(sk.decode_attention(layer, q))
    k_in, v_in = f64(layer.k), f64(layer.v)
    empty = [b for b in range(B) if int(lens[b]) == 0]
    assert empty and all(not out[b].any() for b in empty)
    for b in [0, 1, 31, 32, 33, 511, 512, 777, 1022, 1023] + [b for b in range(B) if int(lens[b]) == 1][:3]:
        rc = rings[b]
        if rc.pos == 0:
            continue
        keys = np.stack([k_in[b][:, s] for s in rc.chronological_slots()])
        vals = np.stack([v_in[b][:, s] for s in rc.chronological_slots()])
        from oracle.sinkkv_oracle import attend
        np.testing.assert_allclose(out[b], attend(f64(q[b]), keys, vals), rtol=0, atol=BF16_ATTN_ATOL)
    big = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1025, 1, D, sinks=S, window=W)
    with pytest.raises(sk.SinkKVError) as e:
        sk.decode_attention(big, torch.zeros(1025, Hq, D, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == sk.SK_ERR_UNSUPPORTED
