"""The allocation-free decode entry point, for callers that cannot call cudaMalloc
(for example a serving loop whose device memory is all carved up by its own pool, or
a plug-in inside a host application that owns every device allocation).

It is checked through the C ABI against the ordinary entry point, which takes a
caller-allocated workspace, on two calls in a row.  This file is collected last so
that a stop-at-first-failure run has already run every other test."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _noalloc(lib, sk, layer, q, out, stream):
    st = layer.struct()
    return lib.sk_decode_attention_noalloc(ctypes.byref(st), ctypes.c_void_p(q.data_ptr()), q.shape[1], sk.SK_BF16,
                                           None, ctypes.c_void_p(out.data_ptr()), stream)


def test_noalloc_decode_matches_workspace_decode_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as sk
    from sink_kv_attention_gb300 import synth
    lib = sk._lib()
    B, Hq, Hkv, D, S, W = 8, 32, 8, 128, 4, 1020
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, B, Hkv, D, sinks=S, window=W)
    synth.fill_normal_(layer.k, 71)
    synth.fill_normal_(layer.v, 72)
    pos, head, count = synth.window_state(73, B, W, 2000, 9000)
    layer.pos.copy_(pos)
    layer.head.copy_(head)
    layer.count.copy_(count)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # First a larger call of another shape whose values are NaN: the shared scratch then
    # holds NaN partials, which the compared calls must never pick up.
    poison = sk.KVLayer.allocate(sk.SK_LAYER_RING, 24, Hkv, D, sinks=S, window=200)
    poison.v.fill_(float("nan"))
    poison.pos.fill_(500)
    poison.count.fill_(200)
    qp = torch.ones(24, Hq, D, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, sk, poison, qp, torch.empty_like(qp), stream) == sk.SK_OK
    for call in range(2):
        q = synth.normal((B, Hq, D), 80 + call, torch.bfloat16).cuda()
        want = sk.decode_attention(layer, q)
        out = torch.full_like(q, float("nan"))
        status = _noalloc(lib, sk, layer, q, out, stream)
        assert status == sk.SK_OK, lib.sk_status_str(status)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: bit for bit the workspace call's output
        assert torch.equal(out, want)
    assert layer.error_bits() == 0


def test_noalloc_decode_rejects_batches_past_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as sk
    lib = sk._lib()
    # 1024 x 8 units need about 17 MB of scratch, past the fixed 4 MiB
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1024, 8, 128, sinks=0, window=1)
    q = torch.zeros(1024, 32, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    st = layer.struct()
    status = lib.sk_decode_attention_noalloc(ctypes.byref(st), ctypes.c_void_p(q.data_ptr()), 32, sk.SK_BF16,
                                             None, ctypes.c_void_p(out.data_ptr()), None)
    assert status == sk.SK_ERR_CAPACITY
