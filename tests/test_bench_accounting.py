"""The bench's work accounting against brute force: the prefill kernel's visited-tile
count (the numerator of its tile-level TFLOP/s) equals the number of 128-row x 64-key
tiles that hold at least one (query, key) pair the oracle's mask admits, for a chunk
alone and for a chunk over a prior cache."""
import numpy as np
import pytest

import bench
from oracle.sinkkv_oracle import mask_allows


def _brute_tiles(T, S, W, n_rep, p0=0, qoff=0, BM=128, BN=64):
    """Tiles with a visible pair: rows are (head, query) of a block of BM // nh queries;
    the key index space is [prior keys, padded to a multiple of BN][chunk keys]
    (positions as the prefill defines; padding has none)."""
    nh = bench._prefill_heads_per_cta(n_rep)
    qpb = BM // nh
    pos = _key_positions(T, S, p0, qoff, BN)
    Tk = len(pos)
    win = W if W > 0 else None
    count = 0
    for q0 in range(0, T, qpb):
        queries = range(q0, min(q0 + qpb, T))
        for k0 in range(0, Tk, BN):
            keys = range(k0, min(k0 + BN, Tk))
            if any(pos[j] is not None and mask_allows(p0 + t, pos[j], S, win) for t in queries for j in keys):
                count += 1
    return count, nh


def _key_positions(T, S, p0, qoff, BN):
    """Absolute position of every key index: the prior's sinks, then its recent keys
    before p0, then padding (None) up to a multiple of BN, then the chunk."""
    if not qoff:
        return list(range(p0, p0 + T))
    s0 = min(S, p0)
    qpad = -(-qoff // BN) * BN
    return (list(range(s0)) + list(range(p0 - (qoff - s0), p0)) + [None] * (qpad - qoff)
            + list(range(p0, p0 + T)))


@pytest.mark.parametrize("T,S,W,n_rep,p0", [
    (300, 4, 100, 4, 0), (300, 0, 100, 4, 0), (300, 4, 0, 4, 0), (513, 3, 130, 1, 1),
    (64, 4, 16, 8, 0), (1000, 4, 300, 2, 0), (257, 4, 1000, 4, 0),
])
def test_prefill_tiles_chunk_alone(T, S, W, n_rep, p0):
    assert bench._prefill_tiles(T, S, W, n_rep, p0=p0) == _brute_tiles(T, S, W, n_rep, p0=p0)


@pytest.mark.parametrize("T,S,W,n_rep,p0", [
    (300, 4, 100, 4, 250), (300, 4, 100, 4, 50), (129, 0, 61, 1, 1000), (260, 3, 300, 8, 700),
    (200, 4, 0, 4, 300), (400, 4, 100, 4, 2), (300, 16, 40, 4, 9),
])
def test_prefill_tiles_chunk_over_prior(T, S, W, n_rep, p0):
    s0 = min(S, p0) if W > 0 else 0
    qoff = s0 + (min(W - 1, p0 - s0) if W > 0 else p0)
    assert bench._prefill_tiles(T, S, W, n_rep, p0=p0, qoff=qoff) == _brute_tiles(T, S, W, n_rep, p0=p0, qoff=qoff)


def _brute_strips(T, S, W, n_rep, p0=0, qoff=0, BM=128, BN=64, strip=16):
    """Query blocks whose key tile 0 holds visible pairs, all of them sink keys that fit in
    one strip: the blocks whose tile 0 the kernel visits as a 16-key strip."""
    nh = bench._prefill_heads_per_cta(n_rep)
    qpb = BM // nh
    pos = _key_positions(T, S, p0, qoff, BN)
    Tk = len(pos)
    win = W if W > 0 else None
    count = 0
    for q0 in range(0, T, qpb):
        pure = []   # tiles below the window: visible keys only as sinks
        for k0 in range(0, Tk, BN):
            pairs = [(t, j) for t in range(q0, min(q0 + qpb, T)) for j in range(k0, min(k0 + BN, Tk))
                     if pos[j] is not None and mask_allows(p0 + t, pos[j], S, win)]
            if pairs and not any(mask_allows(p0 + t, pos[j], 0, win) for t, j in pairs):
                pure.append((k0, max(j for _, j in pairs)))
        # tile 0 is the one tile of sinks alone, and its sinks fit in a strip
        if W > 0 and len(pure) == 1 and pure[0][0] == 0 and pure[0][1] < strip:
            count += 1
    return count


@pytest.mark.parametrize("T,S,W,n_rep,p0,qoff", [
    (300, 4, 100, 4, 0, 0), (300, 0, 100, 4, 0, 0), (300, 4, 0, 4, 0, 0), (513, 3, 130, 1, 1, 0),
    (1000, 4, 300, 2, 0, 0), (700, 20, 100, 4, 0, 0), (300, 4, 100, 4, 250, 103), (400, 4, 100, 4, 2, 2),
])
def test_prefill_sink_strips(T, S, W, n_rep, p0, qoff):
    assert (bench._prefill_tiles(T, S, W, n_rep, p0=p0, qoff=qoff, strips=True)[2]
            == _brute_strips(T, S, W, n_rep, p0=p0, qoff=qoff))


def test_every_bench_row_times_the_oracle_beside_it():
    """Each row of the default run carries an oracle baseline: a timed CPU function
    exists for every row name."""
    assert {name for name, _ in bench.ROWS} <= set(bench.CPU_ROWS)


@pytest.mark.parametrize("row", ["window_step", "window_i8", "paged"])
def test_single_sequence_oracle_baselines_run(row, monkeypatch):
    """The oracle baselines of the decode-step, int8-key and paged rows run on the host
    and report the row's unit (a minimal sample)."""
    monkeypatch.setattr(bench, "CPU_ROW_SECS", 0.0)
    r = bench.CPU_ROWS[row]()
    assert r["unit"] == "GB/s" and r["value"] > 0 and "extrapolated" in r["sample"]
