"""Host-side pieces of the library, run without a GPU: the cos/sin table build on host
threads and the dynamic YaRN factor policy, against the float64 oracle and the
values the pages print."""
import numpy as np
import pytest

from oracle.sinkkv_oracle import RopeSpec, dynamic_factor as o_dynamic_factor, rope_table
from tests.conftest import golden_path


@pytest.fixture(scope="module")
def sk():
    import os
    import sink_kv_attention_gb300 as m
    if not os.path.exists(m.LIB_PATH):
        from sink_kv_attention_gb300 import build
        build.build()
    m._lib()
    return m


@pytest.mark.parametrize("factor", [1.0, 1.125, 2.0])
def test_threaded_table_build_is_bitwise_the_single_thread_build(sk, factor):
    """"#2961 rope: --rope-scaling dynamic", "Measured on this branch": the threaded
    build equals the single-thread one bit for bit (factors 1, 1.125, 2; 1, 7 and 16
    threads)."""
    args = dict(head_dim=128, rotary_dim=64, theta=5e5, max_positions=20011, yarn_factor=factor,
                yarn_orig_ctx=8192)
    one = sk.rope_table_fill_host(**args, n_threads=1)
    for n in (7, 16, 0):
        assert np.array_equal(sk.rope_table_fill_host(**args, n_threads=n).view(np.uint32), one.view(np.uint32))


@pytest.mark.parametrize("neox,factor,theta,r", [(True, 1.0, 1e4, 128), (True, 2.0, 5e5, 64),
                                                 (False, 8.0, 1e4, 128), (True, 1.5, 5e5, 64)])
def test_host_table_matches_oracle_rounded_to_float32(sk, neox, factor, theta, r):
    """Every entry within one float32 ulp of the oracle's float64 mu (cos, sin)(P w_j),
    plus what a few float64 ulps of difference in the angle P w_j can move a value
    near a zero of cos or sin; nearly all bitwise."""
    n = 9000
    got = sk.rope_table_fill_host(128, r, theta, n, neox=neox, yarn_factor=factor, yarn_orig_ctx=4096)
    spec = RopeSpec(128, r, theta, neox, factor, 4096)
    want64 = rope_table(spec, n)
    want = want64.astype(np.float32)
    ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
    angle = np.arange(n, dtype=np.float64)[:, None] * spec.omega()[None, :]
    tol = ulp + spec.mscale() * angle[..., None] * 1e-15
    diff = np.abs(got.astype(np.float64) - want.astype(np.float64))
    assert np.all(diff <= tol), float((diff / tol).max())
    assert np.mean(diff == 0) > 0.99


def test_host_table_rejects_bad_arguments(sk):
    import ctypes
    lib = sk._lib()
    buf = np.zeros(64, dtype=np.float32)
    bad = sk.RopeConfig(128, 72, 1, 0, 1e4, 1.0, 4096, 32.0, 1.0, 1)
    assert lib.sk_rope_table_fill_host(ctypes.byref(bad), 0, buf.ctypes.data_as(ctypes.c_void_p)) == sk.SK_ERR_ARG
    good = sk.RopeConfig(128, 64, 1, 0, 1e4, 1.0, 4096, 32.0, 1.0, 1)
    assert lib.sk_rope_table_fill_host(ctypes.byref(good), -1, buf.ctypes.data_as(ctypes.c_void_p)) == sk.SK_ERR_ARG
    assert lib.sk_rope_table_fill_host(ctypes.byref(good), 0, None) == sk.SK_ERR_ARG


def _factor_golden():
    rows = []
    with open(golden_path("dynamic_factor_values.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                t, L0, step, cap, want = line.split()
                rows.append((int(t), int(L0), float(step), float(cap), float(want)))
    return rows


def test_dynamic_factor_reproduces_page_values(sk):
    rows = _factor_golden()
    assert rows
    for t, L0, step, cap, want in rows:
        assert sk.dynamic_factor(t, L0, step, cap) == want, (t, L0)


def test_dynamic_factor_equals_oracle_over_a_sweep(sk):
    rng = np.random.default_rng(5)
    for L0 in (4096, 8100, 262144):
        totals = np.concatenate([np.arange(L0 - 3, L0 + 5), rng.integers(0, 3 * L0, 400),
                                 (L0 * np.arange(1, 17) / 8).astype(np.int64)])
        for t in totals:
            for step, cap in ((0.125, 2.0), (0.25, 3.0), (0.1, 8.0)):
                assert sk.dynamic_factor(int(t), L0, step, cap) == o_dynamic_factor(int(t), L0, step, cap)


def test_dynamic_factor_page_chain_of_switches(sk):
    """The lengths at which a dialog crosses into each factor of the page's chain
    1 -> 1.125 -> 1.25 -> 1.5 -> 1.625 -> 1.75 -> 1.875 -> 2 (L0 = 262,144)."""
    L0 = 262144
    chain = [1.0, 1.125, 1.25, 1.5, 1.625, 1.75, 1.875, 2.0]
    for f in chain[1:]:
        first = int(np.floor(L0 * (f - 0.125))) + 1   # first length that needs factor f
        assert sk.dynamic_factor(first, L0) == f
        assert sk.dynamic_factor(first - 1, L0) == f - 0.125


def test_dynamic_factor_rejects_bad_arguments(sk):
    import ctypes
    lib = sk._lib()
    f = ctypes.c_double()
    assert lib.sk_rope_dynamic_factor(-1, 4096, 0.125, 2.0, ctypes.byref(f)) == sk.SK_ERR_ARG
    assert lib.sk_rope_dynamic_factor(10, 0, 0.125, 2.0, ctypes.byref(f)) == sk.SK_ERR_ARG
    assert lib.sk_rope_dynamic_factor(10, 4096, 0.0, 2.0, ctypes.byref(f)) == sk.SK_ERR_ARG
    assert lib.sk_rope_dynamic_factor(10, 4096, 0.125, 0.5, ctypes.byref(f)) == sk.SK_ERR_ARG
    assert lib.sk_rope_dynamic_factor(10, 4096, 0.125, 2.0, None) == sk.SK_ERR_ARG
