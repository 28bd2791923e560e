"""Failure detection on the GPU without a fault: an in-kernel wait that can never be
satisfied gives up after its limit, reports SK_DEVERR_TIMEOUT through the device error
word, and the context keeps working.  The same for the prefill pipeline, whose softmax
warps are told (by the self-test entry point) never to signal one tile's P: the blocks
that reach it stop every role, drain what they issued and report."""
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


def _chunk(T, seed):
    from sink_kv_attention_gb300 import synth
    q = synth.normal((1, T, 8, 128), seed, torch.bfloat16, device="cuda")
    k = synth.normal((1, T, 2, 128), seed + 1, torch.bfloat16, device="cuda")
    v = synth.normal((1, T, 2, 128), seed + 2, torch.bfloat16, device="cuda")
    return q, k, v


def test_prefill_stall_times_out_drains_and_reports(sk):
    # T = 512, 4 q heads per block (32 queries), causal: blocks 4..15 of each head group
    # visit 3 or more key tiles and stall at tile 2; blocks 0..3 finish normally
    q, k, v = _chunk(512, 31)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    sk.selftest_prefill_stall(q, k, v, 2, err)
    status, bits = sk.sync_check(err, clear=True)
    elapsed = time.perf_counter() - t0
    assert bits == sk.SK_DEVERR_TIMEOUT and status == sk.SK_ERR_CUDA
    # every stalled block gives up after one wait's limit (the roles stop together),
    # not after one limit per remaining wait
    assert 0.9 < elapsed < 10.0
    # the context is still usable and the kernel still right: a normal call afterwards
    # equals a fresh one bit for bit and reports nothing
    a = sk.prefill_attention(q, k, v, 0, 0, 0, err=err)
    b = sk.prefill_attention(q, k, v, 0, 0, 0, err=err)
    status, bits = sk.sync_check(err, clear=True)
    assert status == sk.SK_OK and bits == 0
    assert torch.equal(a, b) and torch.isfinite(a.float()).all()


def test_prefill_stall_past_every_tile_changes_nothing(sk):
    # a stall tile no block reaches: the pipeline runs as the product call does
    q, k, v = _chunk(512, 37)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = sk.selftest_prefill_stall(q, k, v, 1 << 20, err)
    want = sk.prefill_attention(q, k, v, 0, 0, 0, err=err)
    status, bits = sk.sync_check(err, clear=True)
    assert status == sk.SK_OK and bits == 0
    assert torch.equal(got, want)
