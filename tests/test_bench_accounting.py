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
    the key index space is [prior keys][chunk keys] (positions as the prefill defines)."""
    nh = bench._prefill_heads_per_cta(n_rep)
    qpb = BM // nh
    Tk = T + qoff
    # absolute positions of the key buffer: sinks, then the recent keys before p0, then the chunk
    if qoff:
        s0 = min(S, p0)
        pos = list(range(s0)) + list(range(p0 - (qoff - s0), p0)) + list(range(p0, p0 + T))
    else:
        pos = list(range(p0, p0 + T))
    win = W if W > 0 else None
    count = 0
    for q0 in range(0, T, qpb):
        queries = range(q0, min(q0 + qpb, T))
        for k0 in range(0, Tk, BN):
            keys = range(k0, min(k0 + BN, Tk))
            if any(mask_allows(p0 + t, pos[j], S, win) for t in queries for j in keys):
                count += 1
    return count, nh


@pytest.mark.parametrize("T,S,W,n_rep,p0", [
    (300, 4, 100, 4, 0), (300, 0, 100, 4, 0), (300, 4, 0, 4, 0), (513, 3, 130, 1, 1),
    (64, 4, 16, 8, 0), (1000, 4, 300, 2, 0), (257, 4, 1000, 4, 0),
])
def test_prefill_tiles_chunk_alone(T, S, W, n_rep, p0):
    assert bench._prefill_tiles(T, S, W, n_rep, p0=p0) == _brute_tiles(T, S, W, n_rep, p0=p0)


@pytest.mark.parametrize("T,S,W,n_rep,p0", [
    (300, 4, 100, 4, 250), (300, 4, 100, 4, 50), (129, 0, 61, 1, 1000), (260, 3, 300, 8, 700),
    (200, 4, 0, 4, 300),
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
    Tk = T + qoff
    if qoff:
        s0 = min(S, p0)
        pos = list(range(s0)) + list(range(p0 - (qoff - s0), p0)) + list(range(p0, p0 + T))
        nsk = S
    else:
        pos = list(range(p0, p0 + T))
        nsk = max(0, S - p0)
    win = W if W > 0 else None
    count = 0
    for q0 in range(0, T, qpb):
        vis = [j for t in range(q0, min(q0 + qpb, T)) for j in range(min(BN, Tk))
               if mask_allows(p0 + t, pos[j], S, win)]
        if vis and W > 0 and max(vis) < nsk and nsk <= strip:
            count += 1
    return count


@pytest.mark.parametrize("T,S,W,n_rep,p0", [
    (300, 4, 100, 4, 0), (300, 0, 100, 4, 0), (300, 4, 0, 4, 0), (513, 3, 130, 1, 1),
    (1000, 4, 300, 2, 0), (700, 20, 100, 4, 0),
])
def test_prefill_sink_strips(T, S, W, n_rep, p0):
    assert bench._prefill_tiles(T, S, W, n_rep, p0=p0, strips=True)[2] == _brute_strips(T, S, W, n_rep, p0=p0)
