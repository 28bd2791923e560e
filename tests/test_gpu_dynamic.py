"""GPU parity: the dynamic YaRN driver ("#2961 rope: --rope-scaling dynamic", "What it
does"): the factor follows the dialog's length, every cached key is turned on a switch
and the live table is rebuilt in place.  The page's chain of seven switches
1 -> 1.125 -> 1.25 -> 1.5 -> 1.625 -> 1.75 -> 1.875 -> 2 is driven by a growing
dialog and checked against the float64 oracle's keys at factor 2."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import RingCache, RopeSpec, attend, dequantize_int8_rows, dynamic_factor, rope_rotate
from tests.test_gpu_rope_append_decode import BF16_ATTN_ATOL, bf16_ulp, f64

pytestmark = pytest.mark.gpu

D, R, THETA, L0, MAXPOS, HKV = 128, 64, 5e5, 4096, 8192, 2
CHAIN = [1.125, 1.25, 1.5, 1.625, 1.75, 1.875, 2.0]


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


def _table_readout(sk, table, neox=True):
    """The table's entries read back through rope_apply of unit pairs (fp32): row P,
    pair j -> (cos, sin) exactly, since the other element of the pair is 0."""
    half = R // 2
    first = np.arange(half) if neox else np.arange(0, R, 2)
    second = first + half if neox else first + 1
    x = torch.zeros(MAXPOS, 1, D, device="cuda")
    x[:, 0, torch.as_tensor(first)] = 1.0
    sk.rope_apply(table, x, torch.arange(MAXPOS, device="cuda"))
    return torch.stack([x[:, 0, torch.as_tensor(first)], x[:, 0, torch.as_tensor(second)]], -1).cpu()


def _lengths():
    """The first dialog length that needs each factor of the chain (1.375 is stepped
    over, as in the page's chain)."""
    out = [int(np.floor(L0 * (f - 0.125))) + 1 for f in CHAIN]
    out[2] = int(np.floor(L0 * 1.375)) + 1        # 5633: straight from 1.25 to 1.5
    return out


def _turns(P, start, lengths):
    """How many switches a key at position P went through after its append."""
    if P < start:
        return len(lengths)
    for i, n in enumerate(lengths):
        if P < n:
            return len(lengths) - 1 - i
    raise AssertionError(P)


@pytest.mark.parametrize("kdt", ["bf16", "i8"])
def test_seven_switch_chain_matches_keys_at_factor_2(sk, kdt):
    from sink_kv_attention_gb300 import synth
    lengths = _lengths()
    assert [dynamic_factor(n, L0, 0.125, 2.0) for n in lengths] == CHAIN
    start, total = 4000, lengths[-1]
    kdtype = torch.bfloat16 if kdt == "bf16" else torch.int8
    dyn = sk.DynamicRope(D, R, THETA, MAXPOS, L0, cap=2.0)
    assert dyn.factor == 1.0
    glob = sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, HKV, D, capacity=total, k_dtype=kdtype)
    ring = sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, HKV, D, sinks=4, window=1000, k_dtype=kdtype)
    layers = [glob, ring]
    raw = synth.uniform((1, total, HKV, D), 90, -1.0, 1.0, torch.bfloat16, device="cuda")
    v = synth.normal((1, total, HKV, D), 91, torch.bfloat16, device="cuda")

    chunks = list(zip([0, start] + lengths[:-1], [start] + lengths))

    def append(table, Ls, a, b):
        for L in Ls:
            sk.kv_append(table, L, None, raw[:, a:b].clone(), v[:, a:b].clone())

    assert dyn.update(start, layers) == (1.0, False)
    append(dyn.table, layers, *chunks[0])
    for (a, n), f in zip(chunks[1:], CHAIN):
        assert dyn.update(n, layers) == (f, True)
        assert dyn.update(n, layers) == (f, False)          # same factor: nothing happens
        append(dyn.table, layers, a, n)
    torch.cuda.synchronize()
    assert all(L.error_bits() == 0 for L in layers)

    # the yardstick: the same keys, in the same chunks, written directly at factor 2
    tB = sk.RopeTable(D, R, THETA, MAXPOS, yarn_factor=2.0, yarn_orig_ctx=L0)
    direct = [sk.KVLayer.allocate(sk.SK_LAYER_GLOBAL, 1, HKV, D, capacity=total, k_dtype=kdtype),
              sk.KVLayer.allocate(sk.SK_LAYER_RING, 1, HKV, D, sinks=4, window=1000, k_dtype=kdtype)]
    for a, n in chunks:
        append(tB, direct, a, n)
    specB = RopeSpec(D, R, THETA, True, 2.0, L0)
    rc = RingCache(4, 1000)
    for a, n in chunks:
        rc.append(list(range(a, n)))
    assert (int(ring.head[0]), int(ring.count[0])) == (rc.head, rc.count)
    ring_slots = [(s, p) for s, p in enumerate(rc.slots) if p is not None]
    raw64 = f64(raw[0])

    def read(L, slots):
        k = L.k[0][:, slots]                                   # [Hkv, n, D]
        if kdt == "bf16":
            return f64(k).transpose(1, 0, 2), None
        sc = L.k_scale[0][:, slots].cpu().numpy()
        return dequantize_int8_rows(k.cpu().numpy(), sc).transpose(1, 0, 2), sc.T

    for L, Ld, slot_pos in [(glob, direct[0], [(p, p) for p in range(total)]), (ring, direct[1], ring_slots)]:
        slots = [s for s, _ in slot_pos]
        pos = np.array([p for _, p in slot_pos])
        exact = rope_rotate(raw64[pos], pos, specB.omega(), specB.mscale(), R)
        turned, _ = read(L, slots)
        written, sc_b = read(Ld, slots)
        # Every rounding (the write and each turn) adds at most half a step per element
        # and a turn mixes the two elements of a pair, so an element's error grows by at
        # most sqrt(2) * 0.5 step per rounding.  The step is that of the row at the time;
        # a turn keeps each pair's norm (times mu_B / mu_A >= 1 here), so no element of
        # any stage exceeds sqrt(2) times the final row max.
        k = np.array([1 + _turns(p, start, lengths) for p in pos])[:, None, None]
        if kdt == "bf16":
            unit = bf16_ulp(np.sqrt(2) * np.abs(exact).max(axis=-1, keepdims=True))
        else:
            unit = np.sqrt(2) * sc_b[:, :, None]
        assert np.all(np.abs(turned - exact) <= k * 0.5 * np.sqrt(2) * unit + 1e-6), \
            float((np.abs(turned - exact) / unit / k).max())
        most = k[:, 0, 0] == 8
        if most.sum() > 100:
            rms_t = np.sqrt(np.mean((turned[most] - exact[most]) ** 2))
            rms_w = np.sqrt(np.mean((written[most] - exact[most]) ** 2))
            assert rms_t / rms_w <= 1.15 * np.sqrt(8), rms_t / rms_w
        # values are never touched
        assert torch.equal(L.v[0][:, slots], Ld.v[0][:, slots])

    # the live table now holds, bit for bit, a fresh build at factor 2
    assert torch.equal(_table_readout(sk, dyn.table), _table_readout(sk, tB))
    # a decode query at factor 2 over the turned global layer
    if kdt == "bf16":
        q = synth.normal((1, 1, 4 * HKV, D), 92, torch.bfloat16, device="cuda")
        q_raw = f64(q[0])
        sk.rope_apply(dyn.table, q[0], torch.tensor([total - 1], device="cuda"))
        out = f64(sk.decode_attention(glob, q[:, 0].contiguous()))[0]
        qr = rope_rotate(q_raw, [total - 1], specB.omega(), specB.mscale(), R)[0]
        keys = rope_rotate(raw64, np.arange(total), specB.omega(), specB.mscale(), R)
        want = attend(qr, keys, f64(v[0]))
        assert float(np.abs(out - want).max()) <= BF16_ATTN_ATOL


def test_back_below_the_trained_context_gives_the_startup_table(sk):
    dyn = sk.DynamicRope(D, R, THETA, MAXPOS, L0, cap=2.0)
    t1 = sk.RopeTable(D, R, THETA, MAXPOS, yarn_factor=1.0, yarn_orig_ctx=L0)
    start = _table_readout(sk, dyn.table)
    assert torch.equal(start, _table_readout(sk, t1))
    assert dyn.update(MAXPOS) == (2.0, True)
    assert not torch.equal(_table_readout(sk, dyn.table), start)
    assert dyn.update(100) == (1.0, True)
    assert torch.equal(_table_readout(sk, dyn.table), start)


def test_table_pointer_is_stable_and_range_is_checked(sk):
    dyn = sk.DynamicRope(D, R, THETA, MAXPOS, L0)   # cap from max_positions / L0 = 2
    ptr = dyn.table.device_ptr()
    assert dyn.update(MAXPOS) == (2.0, True)
    assert dyn.table.device_ptr() == ptr
    with pytest.raises(sk.SinkKVError) as e:
        dyn.update(MAXPOS + 1)
    assert e.value.status == sk.SK_ERR_POSITION_RANGE
    assert dyn.factor == 2.0
