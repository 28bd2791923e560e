"""The hot path runs inside a captured CUDA graph exactly as it runs eagerly: all state
lives on the device, so a replay of captured append + decode steps gives the same bits
as the same calls launched one by one (also across two streams with their own
workspaces)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def _layer(sk, seed):
    from sink_kv_attention_gb300 import synth
    B, Hkv, D, S, W = 8, 2, 128, 4, 500
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, seed)
    synth.fill_normal_(layer.v, seed + 1)
    pos, head, count = synth.window_state(seed + 2, B, W, 600, 3000)
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    return layer


def _clone(sk, layer):
    return sk.KVLayer(**{f: (getattr(layer, f).clone() if torch.is_tensor(getattr(layer, f)) else getattr(layer, f))
                         for f in layer.__dataclass_fields__})


def test_captured_steps_equal_eager_steps(sk):
    from sink_kv_attention_gb300 import synth
    steps, B, Hq, Hkv, D = 6, 8, 8, 2, 128
    tbl = sk.RopeTable(D, D, 5e5, 4096)
    a = _layer(sk, 70)
    b = _clone(sk, a)
    qs = synth.normal((steps, B, 1, Hq, D), 71, torch.bfloat16, device="cuda")
    ks = synth.normal((steps, B, 1, Hkv, D), 72, torch.bfloat16, device="cuda")
    vs = synth.normal((steps, B, 1, Hkv, D), 73, torch.bfloat16, device="cuda")
    z = torch.linspace(-3.0, 3.0, Hq, device="cuda")
    # eager
    qa, ka, va = qs.clone(), ks.clone(), vs.clone()
    outs_a = []
    for i in range(steps):
        sk.kv_append(tbl, a, qa[i], ka[i], va[i])
        outs_a.append(sk.decode_attention(a, qa[i, :, 0], sink_logits=z).clone())
    # captured
    qb, kb, vb = qs.clone(), ks.clone(), vs.clone()
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    outs_b = torch.empty(steps, B, Hq, D, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(sk.decode_workspace_bytes(b, Hq), dtype=torch.uint8, device="cuda")
    sk.decode_attention(_clone(sk, b), qb[0, :, 0].clone(), out=out, workspace=ws)  # first-use set-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(steps):
            sk.kv_append(tbl, b, qb[i], kb[i], vb[i])
            sk.decode_attention(b, qb[i, :, 0], out=out, workspace=ws, sink_logits=z)
            outs_b[i].copy_(out)
    g.replay()
    torch.cuda.synchronize()
    for i in range(steps):
        assert torch.equal(outs_a[i], outs_b[i]), i
    for f in ("k", "v", "pos", "head", "count"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    assert a.error_bits() == 0 and b.error_bits() == 0


def test_two_streams_with_own_workspaces(sk):
    """Two layers decoded concurrently on two streams, each with its own workspace,
    give the same bits as one after the other."""
    from sink_kv_attention_gb300 import synth
    B, Hq, D = 8, 8, 128
    l1, l2 = _layer(sk, 80), _layer(sk, 90)
    q1 = synth.normal((B, Hq, D), 81, torch.bfloat16, device="cuda")
    q2 = synth.normal((B, Hq, D), 91, torch.bfloat16, device="cuda")
    want1 = sk.decode_attention(l1, q1)
    want2 = sk.decode_attention(l2, q2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    w1 = torch.empty(sk.decode_workspace_bytes(l1, Hq), dtype=torch.uint8, device="cuda")
    w2 = torch.empty(sk.decode_workspace_bytes(l2, Hq), dtype=torch.uint8, device="cuda")
    o1, o2 = torch.empty_like(q1), torch.empty_like(q2)
    torch.cuda.synchronize()
    for _ in range(5):
        with torch.cuda.stream(s1):
            sk.decode_attention(l1, q1, out=o1, workspace=w1, stream=s1)
        with torch.cuda.stream(s2):
            sk.decode_attention(l2, q2, out=o2, workspace=w2, stream=s2)
    torch.cuda.synchronize()
    assert torch.equal(o1, want1) and torch.equal(o2, want2)


def test_captured_chunked_prefill_equals_eager(sk):
    """Chunks of a prompt (rotate, attend over the prior ring, append the rotated keys)
    captured as one graph give the same bits as the same calls made eagerly."""
    from sink_kv_attention_gb300 import synth
    B, Hq, Hkv, D, S, W, T, n = 2, 8, 2, 128, 4, 200, 96, 3
    tbl = sk.RopeTable(D, D, 1e4, 4096)
    q = synth.normal((n, B, T, Hq, D), 90, torch.bfloat16, device="cuda")
    k = synth.normal((n, B, T, Hkv, D), 91, torch.bfloat16, device="cuda")
    v = synth.normal((n, B, T, Hkv, D), 92, torch.bfloat16, device="cuda")
    p_first = 300  # the first chunk starts after a prompt already in the cache

    def fresh():
        layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
        synth.fill_normal_(layer.k, 93)
        synth.fill_normal_(layer.v, 94)
        layer.pos.fill_(p_first)
        layer.count.fill_(W)
        layer.head.fill_(17)
        return layer

    ws = torch.empty(sk.prefill_workspace_bytes(B, T, Hkv, D, sk.prefill_prior_keys(p_first + n * T, S, W)),
                     dtype=torch.uint8, device="cuda")
    posn = [torch.arange(p_first + i * T, p_first + (i + 1) * T, dtype=torch.int64, device="cuda").repeat(B)
            for i in range(n)]

    def run(layer, qs, ks, outs):
        for i in range(n):
            sk.rope_apply(tbl, qs[i].view(B * T, Hq, D), posn[i])
            sk.rope_apply(tbl, ks[i].view(B * T, Hkv, D), posn[i])
            sk.prefill_attention(qs[i], ks[i], v[i], p_first + i * T, S, W, out=outs[i], workspace=ws,
                                 prior=layer, err=layer.err)
            sk.kv_append(None, layer, None, ks[i], v[i])

    eager, qe, ke = fresh(), q.clone(), k.clone()
    out_e = torch.empty(n, B, T, Hq, D, dtype=torch.bfloat16, device="cuda")
    run(eager, qe, ke, out_e)
    torch.cuda.synchronize()
    graph_layer, qg, kg = fresh(), q.clone(), k.clone()
    out_g = torch.empty_like(out_e)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(graph_layer, qg, kg, out_g)
    graph_layer2 = fresh()  # capture does not run: replay on fresh state and inputs
    for f in ("k", "v", "pos", "head", "count"):
        getattr(graph_layer, f).copy_(getattr(graph_layer2, f))
    qg.copy_(q)
    kg.copy_(k)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_e)
    assert torch.equal(graph_layer.k, eager.k) and torch.equal(graph_layer.v, eager.v)
    assert graph_layer.pos.tolist() == eager.pos.tolist() == [p_first + n * T] * B
    assert graph_layer.head.tolist() == eager.head.tolist()
    assert eager.error_bits() == 0 and graph_layer.error_bits() == 0
