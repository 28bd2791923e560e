"""GPU parity of the decode step (sk_decode_step: RoPE + append + attention in two
kernels).  Against the same step taken as sk_kv_append + sk_decode_attention on a copy
of the layer, bit for bit: outputs, cache rows, ring state and error word, over ring
and global layers in every state the append's rules tell apart (sink slots, a ring
filling, a full ring at any head, a one-slot window, a full global layer, a position
past the table), three steps in a row, with and without a table and learned sinks, and
inside a CUDA graph.  Against the float64 oracle at the windowed workload's size, with
probe heads that see every key."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import RopeSpec, decode_attention as o_decode, rope_rotate
from sink_kv_attention_gb300 import synth
from tests.test_gpu_fullsize_keys import DENSITY, _ring_mirror_from_inputs, assert_exact_mean
from tests.test_gpu_rope_append_decode import BF16_ATTN_ATOL, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def _clone(sk, L):
    c = lambda t: None if t is None else t.clone()
    return sk.KVLayer(L.kind, L.k.clone(), L.v.clone(), L.pos.clone(), L.sinks, L.window, c(L.head), c(L.count),
                      c(L.k_scale), c(L.err))


def _assert_same_layer(a, b):
    assert torch.equal(a.k, b.k)
    assert torch.equal(a.v, b.v)
    assert torch.equal(a.pos, b.pos)
    if a.head is not None:
        assert torch.equal(a.head, b.head)
        assert torch.equal(a.count, b.count)
    assert torch.equal(a.err, b.err)


def _both_paths(sk, table, layer, q, k, v, sink_logits=None):
    """The step on a copy of `layer` as kv_append + decode_attention, and on `layer` as
    decode_step; returns (the copy, decode_step's output, the two-call output)."""
    ref = _clone(sk, layer)
    qa, ka = q.clone().unsqueeze(1), k.clone().unsqueeze(1)  # [B, 1, H, D]
    sk.kv_append(table, ref, qa if table is not None else None, ka, v.unsqueeze(1).contiguous())
    want = sk.decode_attention(ref, qa[:, 0].contiguous() if table is not None else q, sink_logits=sink_logits)
    q0, k0, v0 = q.clone(), k.clone(), v.clone()
    got = sk.decode_step(table, layer, q, k, v, sink_logits=sink_logits)
    assert torch.equal(q, q0) and torch.equal(k, k0) and torch.equal(v, v0)  # read only
    return ref, got, want


def _ring(sk, dtype, B, Hkv, D, S, W, states, seed):
    """A ring layer with random rows and per-sequence (pos, head, count)."""
    L = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W, k_dtype=dtype, v_dtype=dtype)
    synth.fill_normal_(L.k, seed)
    synth.fill_normal_(L.v, seed + 1)
    L.pos.copy_(torch.tensor([s[0] for s in states], dtype=torch.int64))
    L.head.copy_(torch.tensor([s[1] for s in states], dtype=torch.int32))
    L.count.copy_(torch.tensor([s[2] for s in states], dtype=torch.int32))
    return L


def _ring_states(S, W):
    """(pos, head, count): the first token, the last sink slot, a ring filling, a full
    ring with the head inside it and at its last slot."""
    st = [(0, 0, 0)]
    st.append((S - 1, 0, 0) if S > 0 else (3, 3 % W, min(3, W)))
    f = min(7, W - 1)
    st.append((S + f, f % W, f))
    st.append((S + W + 123, 123 % W, W))
    st.append((S + 5 * W + W - 1, W - 1, W))
    return st


RING_CASES = [
    # dtype, D, r, neox, Hq, Hkv, S, W
    (torch.bfloat16, 128, 128, True, 32, 8, 4, 300),
    (torch.bfloat16, 128, 64, False, 8, 4, 4, 300),
    (torch.bfloat16, 64, 64, True, 16, 2, 0, 100),
    (torch.float32, 128, 128, False, 4, 4, 2, 50),
    (torch.float32, 64, 32, True, 8, 2, 4, 1),
]


@pytest.mark.parametrize("case", RING_CASES)
def test_ring_step_is_append_then_decode(sk, case):
    dtype, D, r, neox, Hq, Hkv, S, W = case
    states = _ring_states(S, W)
    B = len(states)
    table = sk.RopeTable(D, r, 5e5, 1 << 20, neox=neox)
    layer = _ring(sk, dtype, B, Hkv, D, S, W, states, 401)
    for step in range(3):
        q = synth.normal((B, Hq, D), 410 + step, dtype).cuda()
        k = synth.normal((B, Hkv, D), 420 + step, dtype).cuda()
        v = synth.normal((B, Hkv, D), 430 + step, dtype).cuda()
        ref, got, want = _both_paths(sk, table, layer, q, k, v)
        assert torch.equal(got, want), step
        _assert_same_layer(layer, ref)
    assert layer.error_bits() == 0


@pytest.mark.parametrize("dtype,D,r,neox,Hq,Hkv,cap", [
    (torch.bfloat16, 128, 64, True, 8, 4, 700),
    (torch.float32, 64, 64, False, 4, 1, 300),
])
def test_global_step_is_append_then_decode(sk, dtype, D, r, neox, Hq, Hkv, cap):
    """Positions 0, 5, two short of the capacity (the third step is refused with
    SK_DEVERR_CAPACITY) and at the capacity (every step refused); a refused sequence
    attends over the rows it has, with q unrotated, in both paths."""
    table = sk.RopeTable(D, r, 1e4, 1 << 20, neox=neox)
    pos = [0, 5, cap - 2, cap]
    B = len(pos)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, D, capacity=cap, k_dtype=dtype, v_dtype=dtype)
    synth.fill_normal_(layer.k, 441)
    synth.fill_normal_(layer.v, 442)
    layer.pos.copy_(torch.tensor(pos, dtype=torch.int64))
    for step in range(3):
        q = synth.normal((B, Hq, D), 450 + step, dtype).cuda()
        k = synth.normal((B, Hkv, D), 460 + step, dtype).cuda()
        v = synth.normal((B, Hkv, D), 470 + step, dtype).cuda()
        ref, got, want = _both_paths(sk, table, layer, q, k, v)
        assert torch.equal(got, want), step
        _assert_same_layer(layer, ref)
    assert layer.error_bits() == sk.SK_DEVERR_CAPACITY
    assert layer.pos.tolist() == [3, 8, cap, cap]


def test_position_past_the_table_is_refused_like_the_append(sk):
    """A table of 520 positions: the sequence at position 519 takes its first step and is
    refused on the second (SK_DEVERR_POSITION_RANGE, state kept, q left unrotated)."""
    D, Hq, Hkv, S, W = 128, 8, 2, 4, 64
    table = sk.RopeTable(D, D, 1e4, 520)
    states = [(100, 32, 64), (519, 67, 64)]
    layer = _ring(sk, torch.bfloat16, 2, Hkv, D, S, W, [(p, h % W, c) for p, h, c in states], 481)
    for step in range(2):
        q = synth.normal((2, Hq, D), 482 + step, torch.bfloat16).cuda()
        k = synth.normal((2, Hkv, D), 484 + step, torch.bfloat16).cuda()
        v = synth.normal((2, Hkv, D), 486 + step, torch.bfloat16).cuda()
        ref, got, want = _both_paths(sk, table, layer, q, k, v)
        assert torch.equal(got, want), step
        _assert_same_layer(layer, ref)
    assert layer.error_bits() == sk.SK_DEVERR_POSITION_RANGE
    assert layer.pos.tolist() == [102, 520]


def test_step_without_table_and_with_learned_sinks(sk):
    """No table: q and k come rotated and are used as given; learned sink logits enter
    in the combine as in the two-call path."""
    D, Hq, Hkv, S, W = 128, 16, 4, 4, 200
    states = _ring_states(S, W)
    B = len(states)
    layer = _ring(sk, torch.bfloat16, B, Hkv, D, S, W, states, 491)
    z = torch.linspace(-12.0, 17.0, Hq).cuda()
    for step in range(2):
        q = synth.normal((B, Hq, D), 492 + step, torch.bfloat16).cuda()
        k = synth.normal((B, Hkv, D), 494 + step, torch.bfloat16).cuda()
        v = synth.normal((B, Hkv, D), 496 + step, torch.bfloat16).cuda()
        ref, got, want = _both_paths(sk, None, layer, q, k, v, sink_logits=z)
        assert torch.equal(got, want), step
        _assert_same_layer(layer, ref)


@pytest.mark.parametrize("kind,B,S,W,cap", [
    ("ring", 64, 4, 8, None),     # 512 units of at most 12 rows: 3-5 units per block
    ("ring", 200, 2, 3, None),    # 1600 units of at most 5 rows: about 50 per block
    ("global", 96, 0, 0, 24),     # 768 units of at most 24 rows
])
def test_many_units_per_block(sk, kind, B, S, W, cap):
    """Blocks that meet many (sequence, kv head) units: the token warp's q ring (two
    slots) wraps many times, its writes of later units wait for the consumers to free a
    slot, and a block writes the token rows of several units.  Random states (filling
    sinks, filling and full rings; global prefixes), three steps, bit for bit."""
    D, Hq, Hkv = 64, 16, 8
    table = sk.RopeTable(D, D, 1e4, 1 << 20)
    g = torch.Generator().manual_seed(B * 7 + W)
    if kind == "ring":
        layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
        pos = torch.randint(0, S + 3 * W, (B,), generator=g)
        cnt = torch.clamp(pos - S, min=0, max=W)
        full = cnt == W
        head = torch.where(full, torch.randint(0, W, (B,), generator=g), cnt % W)
        layer.pos.copy_(pos)
        layer.count.copy_(cnt.to(torch.int32))
        layer.head.copy_(head.to(torch.int32))
    else:
        layer = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, B, Hkv, D, capacity=cap)
        layer.pos.copy_(torch.randint(0, cap - 3, (B,), generator=g))
    synth.fill_normal_(layer.k, 601)
    synth.fill_normal_(layer.v, 602)
    for step in range(3):
        q = synth.normal((B, Hq, D), 610 + step, torch.bfloat16).cuda()
        k = synth.normal((B, Hkv, D), 620 + step, torch.bfloat16).cuda()
        v = synth.normal((B, Hkv, D), 630 + step, torch.bfloat16).cuda()
        ref, got, want = _both_paths(sk, table, layer, q, k, v)
        assert torch.equal(got, want), step
        _assert_same_layer(layer, ref)
    assert layer.error_bits() == 0


def test_step_in_a_cuda_graph(sk):
    """Three steps through two layers captured in one CUDA graph and replayed: the same
    bits as the steps taken eagerly (the state changes on the device, at replay)."""
    D, Hq, Hkv, S, W, B = 128, 32, 8, 4, 500, 3
    table = sk.RopeTable(D, D, 5e5, 1 << 20)
    states = [(20, 16, 16), (S + W + 40, 40, W), (S + 3 * W + W - 1, W - 1, W)]
    layers = [_ring(sk, torch.bfloat16, B, Hkv, D, S, W, states, 501 + 10 * i) for i in range(2)]
    eager = [_clone(sk, L) for L in layers]
    qs = [synth.normal((B, Hq, D), 520 + i, torch.bfloat16).cuda() for i in range(6)]
    ks = [synth.normal((B, Hkv, D), 530 + i, torch.bfloat16).cuda() for i in range(6)]
    vs = [synth.normal((B, Hkv, D), 540 + i, torch.bfloat16).cuda() for i in range(6)]
    ws = torch.empty(sk.decode_step_workspace_bytes(layers[0], Hq), dtype=torch.uint8, device="cuda")
    outs = [torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda") for _ in range(6)]
    want = [sk.decode_step(table, eager[i % 2], qs[i], ks[i], vs[i]) for i in range(6)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):  # capture runs nothing: the layers are still as created
        for i in range(6):
            sk.decode_step(table, layers[i % 2], qs[i], ks[i], vs[i], out=outs[i], workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    for i in range(6):
        assert torch.equal(outs[i], want[i]), i
    for L, E in zip(layers, eager):
        _assert_same_layer(L, E)


@pytest.mark.parametrize("B", [1, 4, 32])
def test_windowed_step_against_the_oracle(sk, B):
    """The windowed workload's shapes (H_q=32, H_kv=8, d_h=128, S=4, W=4092, full rings at
    random heads) through decode_step, against the oracle's append + decode: heads
    h % 4 == 0 are probes (q = 0, V sparse signs: the output is the exact mean of every
    visible V row, the new one included), the others within the bf16 tolerance."""
    c = synth.WINDOW
    Hq, Hkv, D, S, W = c["Hq"], c["Hkv"], c["D"], c["S"], c["W"]
    nrep = Hq // Hkv
    tbl = sk.RopeTable(D, c["r"], c["theta"], c["pos_hi"] + 2)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 551 + B)
    synth.fill_sparse_signs_(layer.v, 552 + B, DENSITY)
    pos, head, count = synth.window_state(553 + B, B, W, c["pos_lo"], c["pos_hi"])
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    k_in, v_in = f64(layer.k), f64(layer.v)
    q = synth.normal((B, Hq, D), 554 + B, torch.bfloat16).cuda()
    q[:, ::nrep] = 0.0
    k = synth.normal((B, Hkv, D), 555 + B, torch.bfloat16).cuda()
    v = synth.sparse_signs((B, Hkv, D), 556 + B, DENSITY).cuda()
    out = f64(sk.decode_step(tbl, layer, q, k, v))
    assert layer.error_bits() == 0
    spec = RopeSpec(D, c["r"], c["theta"])
    rand = [h for h in range(Hq) if h % nrep]
    for b in range(B):
        P = int(pos[b])
        ring = _ring_mirror_from_inputs(S, W, P, head[b], count[b], k_in[b], v_in[b])
        qr = rope_rotate(f64(q[b])[None], [P], spec.omega(), 1.0, D)[0]
        kr = rope_rotate(f64(k[b])[None], [P], spec.omega(), 1.0, D)[0]
        ring.append([(kr, f64(v[b]))])
        want = o_decode(ring, qr)
        assert_exact_mean(out[b, ::nrep], want[::nrep], S + W)
        assert float(np.abs(out[b, rand] - want[rand]).max()) <= BF16_ATTN_ATOL
    assert layer.pos.tolist() == [int(x) + 1 for x in pos]
    assert layer.count.tolist() == [W] * B
    assert layer.head.tolist() == [(int(h) + 1) % W for h in head]


def test_step_refuses_a_table_of_another_head_dim(sk):
    """A table built for d_h = 64 against a d_h = 128 layer: SK_ERR_ARG, nothing launched,
    the state as it was."""
    table = sk.RopeTable(64, 64, 1e4, 1024)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, 2, 128, sinks=4, window=16)
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sk.SinkKVError):
        sk.decode_step(table, layer, q, k, k.clone())
    assert layer.pos.tolist() == [0] and layer.error_bits() == 0
