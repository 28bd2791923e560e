"""Zero-length calls through the binding: appending, rotating or attending over a
chunk of no tokens (empty tensors, whose data pointers are NULL) changes nothing and
raises nothing; the cache still decodes as before."""
import pytest
import torch

from sink_kv_attention_gb300 import synth

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def _empty(*shape):
    return torch.empty(*shape, dtype=torch.bfloat16, device="cuda")


def test_zero_token_calls_change_nothing(sk):
    B, Hq, Hkv, S, W = 2, 8, 2, 4, 60
    tbl = sk.RopeTable(D, D, 1e4, 4096)
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    sk.kv_append(tbl, layer, synth.normal((B, 100, Hq, D), 90, torch.bfloat16).cuda(),
                 synth.normal((B, 100, Hkv, D), 91, torch.bfloat16).cuda(),
                 synth.normal((B, 100, Hkv, D), 92, torch.bfloat16).cuda())
    q = synth.normal((B, Hq, D), 93, torch.bfloat16, device="cuda")
    before = sk.decode_attention(layer, q)
    state = [t.clone() for t in (layer.k, layer.v, layer.pos, layer.head, layer.count)]

    sk.kv_append(tbl, layer, _empty(B, 0, Hq, D), _empty(B, 0, Hkv, D), _empty(B, 0, Hkv, D))
    sk.kv_append(None, layer, None, _empty(B, 0, Hkv, D), _empty(B, 0, Hkv, D))
    x = _empty(0, Hq, D)
    sk.rope_apply(tbl, x, torch.empty(0, dtype=torch.int64, device="cuda"))
    out = sk.prefill_attention(_empty(B, 0, Hq, D), _empty(B, 0, Hkv, D), _empty(B, 0, Hkv, D), 100, S, W)
    assert out.shape == (B, 0, Hq, D)
    out = sk.prefill_attention(_empty(B, 0, Hq, D), _empty(B, 0, Hkv, D), _empty(B, 0, Hkv, D), 100, S, W,
                               prior=layer, err=layer.err)
    assert out.shape == (B, 0, Hq, D)
    torch.cuda.synchronize()

    for a, b in zip(state, (layer.k, layer.v, layer.pos, layer.head, layer.count)):
        assert torch.equal(a, b)
    assert layer.error_bits() == 0
    assert torch.equal(sk.decode_attention(layer, q), before)


def test_zero_token_paged_append(sk):
    B, Hkv = 2, 2
    tbl = sk.RopeTable(D, D, 1e4, 4096)
    layer = sk.PagedLayer.allocate(B, Hkv, D, block_size=16, n_blocks=8, max_blocks=4)
    lens = layer.seq_lens.clone()
    sk.paged_append(tbl, layer, None, _empty(B, 0, Hkv, D), _empty(B, 0, Hkv, D))
    torch.cuda.synchronize()
    assert torch.equal(layer.seq_lens, lens)
    assert layer.error_bits() == 0
