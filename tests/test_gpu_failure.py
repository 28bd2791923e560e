"""Failure detection on the GPU without a fault: an in-kernel wait that can never be
satisfied gives up after its limit, reports SK_DEVERR_TIMEOUT through the device error
word, and the context keeps working."""
import time

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


def test_unsatisfiable_wait_times_out_and_reports(sk):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    sk.selftest_bounded_wait(err)
    status, bits = sk.sync_check(err, clear=True)
    elapsed = time.perf_counter() - t0
    assert bits == sk.SK_DEVERR_TIMEOUT and status == sk.SK_ERR_CUDA
    assert 0.9 < elapsed < 30.0  # the wait's limit is about one second
    assert int(err.item()) == 0  # cleared
    # the context is still usable: a decode step right after matches a second one bit for bit
    from sink_kv_attention_gb300 import synth
    layer = sk.KVLayer.allocate(sk.SK_LAYER_RING, 2, 2, 128, sinks=2, window=30)
    synth.fill_normal_(layer.k, 3)
    synth.fill_normal_(layer.v, 4)
    layer.pos.fill_(40)
    layer.count.fill_(30)
    q = synth.normal((2, 8, 128), 5, torch.bfloat16, device="cuda")
    a = sk.decode_attention(layer, q)
    b = sk.decode_attention(layer, q)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.isfinite(a.float()).all()
    assert layer.error_bits() == 0


def test_selftest_argument_check(sk):
    assert sk._lib().sk_selftest_bounded_wait(None, None) == sk.SK_ERR_ARG
