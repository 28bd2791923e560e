"""The C-ABI library loads and exports every symbol include/sinkkv.h declares, and its
host-side argument checks reject bad calls before touching the GPU (no compute calls)."""
import ctypes
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "sinkkv.h")


def _declared():
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^SK_API\s+[\w\s\*]+?\b(sk_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import sink_kv_attention_gb300 as sk
    if not os.path.exists(sk.LIB_PATH):
        from sink_kv_attention_gb300 import build
        build.build()
    return sk._lib()


def test_header_declares_the_five_operations():
    names = _declared()
    for op in ["sk_rope_apply", "sk_kv_append", "sk_decode_attention", "sk_prefill_attention",
               "sk_kv_rerotate", "sk_rope_table_create", "sk_rope_table_rebuild"]:
        assert op in names


def test_library_exports_every_declared_symbol(lib):
    import sink_kv_attention_gb300 as sk
    declared = _declared()
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(sk.EXPORTED) == declared
    out = subprocess.run(["nm", "-D", "--defined-only", sk.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted(l.split()[-1] for l in out.splitlines() if " T " in l)
    assert exported == declared  # nothing else leaks out of the library


def test_status_strings_and_version(lib):
    assert lib.sk_status_str(0) == b"SK_OK"
    assert b"capacity" in lib.sk_status_str(2)
    assert lib.sk_version() >= 100


def test_struct_layouts_match_header(tmp_path):
    """ctypes mirrors of sk_rope_config / sk_kv_layer / sk_paged_layer match the C
    compiler's layout."""
    import sink_kv_attention_gb300 as sk
    src = tmp_path / "layout.c"
    fields = {"sk_rope_config": [f for f, _ in sk.RopeConfig._fields_],
              "sk_kv_layer": [f for f, _ in sk.KVLayerStruct._fields_],
              "sk_paged_layer": [f for f, _ in sk.PagedLayerStruct._fields_]}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "sinkkv.h"', "int main(void) {"]
    for st, fs in fields.items():
        lines.append(f'printf("{st} %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'printf("{st}.{f} %zu\\n", offsetof({st}, {f}));')
    lines.append("return 0; }")
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True).stdout.splitlines())
    for name, cls in [("sk_rope_config", sk.RopeConfig), ("sk_kv_layer", sk.KVLayerStruct),
                      ("sk_paged_layer", sk.PagedLayerStruct)]:
        assert int(got[name]) == ctypes.sizeof(cls)
        for f, _ in cls._fields_:
            assert int(got[f"{name}.{f}"]) == getattr(cls, f).offset, f


def test_bad_arguments_rejected_on_host(lib):
    import sink_kv_attention_gb300 as sk
    out = ctypes.c_void_p()
    bad = sk.RopeConfig(96, 64, 1, 0, 1e4, 1.0, 4096, 32.0, 1.0, 16)   # head_dim 96 unsupported
    assert lib.sk_rope_table_create(ctypes.byref(bad), None, ctypes.byref(out)) == sk.SK_ERR_ARG
    bad = sk.RopeConfig(128, 72, 1, 0, 1e4, 1.0, 4096, 32.0, 1.0, 16)  # r not a multiple of 16
    assert lib.sk_rope_table_create(ctypes.byref(bad), None, ctypes.byref(out)) == sk.SK_ERR_ARG
    bad = sk.RopeConfig(128, 128, 1, 0, 1.0, 1.0, 4096, 32.0, 1.0, 16)  # theta must exceed 1
    assert lib.sk_rope_table_create(ctypes.byref(bad), None, ctypes.byref(out)) == sk.SK_ERR_ARG
    assert lib.sk_rope_table_create(None, None, ctypes.byref(out)) == sk.SK_ERR_ARG
    assert lib.sk_kv_append(None, None, None, 0, None, None, 0, 1, None) == sk.SK_ERR_ARG
    assert lib.sk_decode_attention(None, None, 8, 0, None, None, None, 0, None) == sk.SK_ERR_ARG
    assert lib.sk_decode_attention_noalloc(None, None, 8, 0, None, None, None) == sk.SK_ERR_ARG
    assert lib.sk_prefill_attention(None, None, None, 1, 1, 1, 1, 128, 0, 0, 0, None, None, None, None, 0, None,
                                    None) == sk.SK_ERR_ARG
    assert lib.sk_decode_workspace_bytes(None, 8) == 0
    assert lib.sk_decode_step(None, None, None, 8, None, None, 0, None, None, None, 0, None) == sk.SK_ERR_ARG
    assert lib.sk_decode_step_workspace_bytes(None, 8) == 0
    assert lib.sk_kv_rerotate(None, 1, None, None, None) == sk.SK_ERR_ARG
    assert lib.sk_rope_apply(None, None, 0, 1, 1, None, None, None) == sk.SK_ERR_ARG
    assert lib.sk_paged_append(None, None, None, 0, None, None, 0, 1, None) == sk.SK_ERR_ARG
    assert lib.sk_paged_decode_attention(None, None, 8, 0, None, None, None, 0, None) == sk.SK_ERR_ARG
    assert lib.sk_paged_decode_workspace_bytes(None, 8) == 0
    bad = sk.PagedLayerStruct(0, 0, 1, 1, 128, 2, 4, 0, 0, 0, 16, 16, 16, 16, None, 16, None)  # block_size 2
    assert lib.sk_paged_decode_workspace_bytes(ctypes.byref(bad), 1) == 0
    assert lib.sk_kv_shift_recent(None, 1, None, -1, None) == sk.SK_ERR_ARG
    lib.sk_rope_table_destroy(None)  # NULL is ignored


def test_decode_step_refusals_on_host(lib):
    """sk_decode_step refuses before any launch: an int8 K cache (its step is the two
    calls), mixed io and cache types, a ring layer without its head array, a misaligned
    q.  The device pointers are never dereferenced on these paths."""
    import sink_kv_attention_gb300 as sk
    A = 1 << 20  # aligned stand-in addresses, never read

    def layer(k_dtype=sk.SK_BF16, head=A + 4096):
        return sk.KVLayerStruct(sk.SK_LAYER_RING, k_dtype, sk.SK_BF16, 2, 8, 128, 4, 60, 64, A, A + 16,
                                A + 32 if k_dtype == sk.SK_I8 else None, head, A + 8192, A + 12288, None)

    def step(L, io=sk.SK_BF16, q=A + 64):
        return lib.sk_decode_step(None, ctypes.byref(L), q, 32, A + 128, A + 256, io, None, A + 512, A + 1024,
                                  1 << 30, None)

    assert step(layer(sk.SK_I8)) == sk.SK_ERR_UNSUPPORTED
    assert lib.sk_decode_step_workspace_bytes(ctypes.byref(layer(sk.SK_I8)), 32) == 0
    assert step(layer(), io=sk.SK_F32) == sk.SK_ERR_UNSUPPORTED
    assert step(layer(head=None)) == sk.SK_ERR_ARG
    assert step(layer(), q=A + 72) == sk.SK_ERR_ARG
    assert lib.sk_decode_step(None, ctypes.byref(layer()), None, 32, A, A, sk.SK_BF16, None, A, A, 1 << 30,
                              None) == sk.SK_ERR_ARG


def test_prefill_prior_keys_are_exactly_the_old_keys_a_chunk_sees(lib):
    """sk_prefill_prior_keys(p0, S, W) is the number of positions before p0 that any
    query of a chunk starting at p0 may see under the oracle's mask (its first query
    sees the most); window <= 0 is a global layer (all of them)."""
    from oracle.sinkkv_oracle import mask_allows
    for p0 in range(0, 40):
        for S in (0, 1, 4):
            for W in (0, 1, 2, 7, 16):
                want = sum(1 for k in range(p0) if mask_allows(p0, k, S, W if W > 0 else None))
                assert lib.sk_prefill_prior_keys(p0, S, W) == want, (p0, S, W)
    assert lib.sk_prefill_prior_keys(-1, 4, 8) == -1
    assert lib.sk_prefill_prior_keys(5, -1, 8) == -1


def test_prefill_workspace_and_prior_arguments_checked_on_host(lib):
    import sink_kv_attention_gb300 as sk
    # no scratch without a prior (a token 16 bytes); with one, the combined keys and values
    assert lib.sk_prefill_workspace_bytes(2, 100, 8, 128, 0) == 16
    # the prior's 30 keys, padded to 64 rows, of K and of V (the chunk is read in place)
    assert lib.sk_prefill_workspace_bytes(2, 100, 8, 128, 30) == 2 * (2 * 64 * 8 * 128 * 2)
    assert lib.sk_prefill_workspace_bytes(2, 100, 8, 128, 64) == 2 * (2 * 64 * 8 * 128 * 2)
    assert lib.sk_prefill_workspace_bytes(2, 100, 8, 128, 65) == 2 * (2 * 128 * 8 * 128 * 2)
    assert lib.sk_prefill_workspace_bytes(2, 100, 8, 128, -1) == 0
    assert lib.sk_prefill_workspace_bytes(2, 100, 8, 64, 0) == 0
    assert lib.sk_prefill_workspace_bytes(2, 0, 8, 128, 30) == 16   # an empty chunk
    assert lib.sk_prefill_workspace_bytes(2, -1, 8, 128, 0) == 0
    fake = 1 << 20  # aligned, never dereferenced: every case below fails before a launch

    def prior(kind=sk.SK_LAYER_RING, k_dtype=sk.SK_BF16, sinks=4, window=60, capacity=64):
        return sk.KVLayerStruct(kind, k_dtype, sk.SK_BF16, 2, 8, 128, sinks, window, capacity, fake, fake, None,
                                fake, fake, fake, None)

    def call(pr, p0=100, sinks=4, window=60, ws=1 << 30):
        return lib.sk_prefill_attention(fake, fake, fake, 2, 100, 32, 8, 128, p0, sinks, window,
                                        ctypes.byref(pr), None, fake, fake, ws, None, None)

    assert call(prior(window=61)) == sk.SK_ERR_ARG                        # ring window differs
    assert call(prior(sinks=2)) == sk.SK_ERR_ARG                          # ring sinks differ
    assert call(prior(), window=0) == sk.SK_ERR_ARG                       # ring under a global mask
    assert call(prior(k_dtype=sk.SK_I8)) == sk.SK_ERR_UNSUPPORTED         # int8 keys
    assert call(prior(kind=sk.SK_LAYER_GLOBAL, capacity=99), window=0) == sk.SK_ERR_CAPACITY
    assert call(prior(), ws=1000) == sk.SK_ERR_ARG                        # workspace too small
    bad = prior()
    bad.batch = 3
    assert call(bad) == sk.SK_ERR_ARG                                     # batch differs


def test_prefill_stall_selftest_arguments_checked_on_host(lib):
    import sink_kv_attention_gb300 as sk
    fake = 1 << 20  # aligned, never dereferenced: every case below fails before a launch

    def call(stall=2, err=fake, T=256, D=128, ws=16):
        return lib.sk_selftest_prefill_stall(fake, fake, fake, 1, T, 8, 2, D, fake, fake, ws, stall, err, None)

    assert call(err=None) == sk.SK_ERR_ARG            # the error word is the test's result
    assert call(stall=-1) == sk.SK_ERR_ARG            # -1 is the product call's "no stall"
    assert call(D=64) == sk.SK_ERR_UNSUPPORTED        # the prefill's own checks apply
    assert call(ws=0) == sk.SK_ERR_ARG
    assert call(T=0) == sk.SK_OK                      # an empty chunk launches nothing


def test_append_without_table_takes_no_q(lib):
    """sk_kv_append with no table appends rotated keys as given; a q would stay
    unrotated, so it is refused on the host (before any launch)."""
    import sink_kv_attention_gb300 as sk
    fake = 1 << 20
    s = sk.KVLayerStruct(sk.SK_LAYER_RING, sk.SK_BF16, sk.SK_BF16, 1, 8, 128, 4, 60, 64, fake, fake, None,
                         fake, fake, fake, None)
    assert lib.sk_kv_append(None, ctypes.byref(s), fake, 32, fake, fake, sk.SK_BF16, 1, None) == sk.SK_ERR_ARG
    s.head_dim = 96
    assert lib.sk_kv_append(None, ctypes.byref(s), None, 0, fake, fake, sk.SK_BF16, 1, None) == \
        sk.SK_ERR_UNSUPPORTED


def test_zero_length_calls_return_ok_without_a_launch(lib):
    """T = 0 passes the host checks and returns SK_OK with nothing launched: the
    pointers below are aligned fakes that a launch would fault on, and no CUDA device
    is needed."""
    import sink_kv_attention_gb300 as sk
    fake = 1 << 20
    s = sk.KVLayerStruct(sk.SK_LAYER_RING, sk.SK_BF16, sk.SK_BF16, 2, 8, 128, 4, 60, 64, fake, fake, None,
                         fake, fake, fake, None)
    assert lib.sk_kv_append(None, ctypes.byref(s), None, 0, fake, fake, sk.SK_BF16, 0, None) == sk.SK_OK
    assert lib.sk_kv_append(None, ctypes.byref(s), None, 0, fake, fake, sk.SK_BF16, -1, None) == sk.SK_ERR_ARG
    assert lib.sk_prefill_attention(fake, fake, fake, 2, 0, 32, 8, 128, 0, 4, 60, None, None, fake, fake, 16,
                                    None, None) == sk.SK_OK
    assert lib.sk_prefill_attention(fake, fake, fake, 2, 0, 32, 8, 128, 100, 4, 60, ctypes.byref(s), None, fake,
                                    fake, 16, None, None) == sk.SK_OK
    assert lib.sk_prefill_attention(fake, fake, fake, 2, -1, 32, 8, 128, 0, 4, 60, None, None, fake, fake, 16,
                                    None, None) == sk.SK_ERR_ARG
    # an empty torch tensor has data_ptr() 0: NULL data pointers are accepted at T = 0 only
    assert lib.sk_kv_append(None, ctypes.byref(s), None, 0, None, None, sk.SK_BF16, 0, None) == sk.SK_OK
    assert lib.sk_kv_append(None, ctypes.byref(s), None, 0, None, None, sk.SK_BF16, 1, None) == sk.SK_ERR_ARG
    assert lib.sk_prefill_attention(None, None, None, 2, 0, 32, 8, 128, 0, 4, 60, None, None, None, None, 0,
                                    None, None) == sk.SK_OK
    assert lib.sk_prefill_attention(None, None, None, 2, 1, 32, 8, 128, 0, 4, 60, None, None, None, None, 0,
                                    None, None) == sk.SK_ERR_ARG
    s.window = 0  # the layer is still checked at T = 0
    assert lib.sk_kv_append(None, ctypes.byref(s), None, 0, None, None, sk.SK_BF16, 0, None) == sk.SK_ERR_ARG
