"""GPU parity: paged KV caches (block tables over a shared pool of blocks, optional
static sink blocks in front of every table): the fused RoPE + paged append and the
split-K decode over 16-token blocks, against the float64 oracle."""
import numpy as np
import pytest
import torch

from oracle.sinkkv_oracle import (RopeSpec, blocks_for_tokens, first_window_token, paged_decode_attention,
                                  rope_rotate, visible_positions)
from tests.test_gpu_rope_append_decode import BF16_ATTN_ATOL, F32_ATTN_ATOL, assert_rows_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sink_kv_attention_gb300 as m
    m._lib()
    return m


class HostAllocator:
    """A test-side block allocator: hands out pool blocks in a shuffled order, frees
    the blocks a window has left behind (their table entries become -1)."""

    def __init__(self, n_blocks, seed, reserved=()):
        rng = np.random.default_rng(seed)
        self.free = [int(b) for b in rng.permutation(n_blocks) if int(b) not in set(reserved)]

    def ensure(self, table, b, n_tokens, bs):
        for j in range(blocks_for_tokens(n_tokens, bs)):
            if table[b, j] < 0:
                table[b, j] = self.free.pop()

    def release_outside(self, table, b, length, bs, sinks, window, sink_len):
        """Free request blocks holding no key the newest query (logical position
        length + sink_len - 1) still sees."""
        if window <= 0:
            return
        keep_lo = first_window_token(length + sink_len - 1, window)
        for j in range(table.shape[1]):
            lo, hi = sink_len + j * bs, sink_len + (j + 1) * bs      # logical keys of request block j
            if table[b, j] >= 0 and hi <= keep_lo and lo >= sinks:
                self.free.append(int(table[b, j]))
                table[b, j] = -1


def _run_paged(sk, *, dtype, D, r, Hq, Hkv, bs, S, W, n_sink_blocks, lengths, chunks, seed, neox=True):
    """Append raw tokens chunk by chunk through the library (allocating blocks before
    each append and freeing those the window left), then decode the last token's
    query; returns everything the oracle needs."""
    from sink_kv_attention_gb300 import synth
    B = len(lengths)
    total = max(lengths)
    sink_len = n_sink_blocks * bs
    max_blocks = blocks_for_tokens(total, bs) + 1
    n_blocks = B * max_blocks + n_sink_blocks + 3
    layer = sk.PagedLayer.allocate(B, Hkv, D, block_size=bs, n_blocks=n_blocks, max_blocks=max_blocks,
                                   sinks=S, window=W, n_sink_blocks=n_sink_blocks, dtype=dtype)
    # static sink blocks: the last n_sink_blocks of the pool, filled with synthetic rotated keys
    sink_ids = list(range(n_blocks - n_sink_blocks, n_blocks))
    sink_k = synth.normal((max(1, n_sink_blocks), Hkv, bs, D), seed + 7, dtype)[:n_sink_blocks]
    sink_v = synth.normal((max(1, n_sink_blocks), Hkv, bs, D), seed + 8, dtype)[:n_sink_blocks]
    if n_sink_blocks:
        layer.sink_block_ids.copy_(torch.tensor(sink_ids, dtype=torch.int32))
        layer.k_pool[sink_ids] = sink_k.cuda()
        layer.v_pool[sink_ids] = sink_v.cuda()
    tbl = sk.RopeTable(D, r, 1e4, total + 8, neox=neox)
    spec = RopeSpec(D, r, 1e4, neox)
    raw_q = synth.normal((B, total, Hq, D), seed, dtype)
    raw_k = synth.normal((B, total, Hkv, D), seed + 1, dtype)
    raw_v = synth.normal((B, total, Hkv, D), seed + 2, dtype)
    alloc = HostAllocator(n_blocks, seed + 3, reserved=sink_ids)
    table = np.full((B, max_blocks), -1, dtype=np.int64)
    done = [0] * B
    q_last = torch.zeros(B, Hq, D, dtype=dtype, device="cuda")
    for T in chunks:
        # every sequence appends T tokens per call (shorter ones stop early: T = 0 calls are skipped)
        active = [b for b in range(B) if done[b] + T <= lengths[b]]
        if not active or T == 0:
            continue
        sub = sk.PagedLayer(layer.k_pool, layer.v_pool, layer.block_table[active].contiguous(),
                            layer.sink_block_ids, layer.seq_lens[active].contiguous(), layer.err, S, W)
        for b in active:
            alloc.ensure(table, b, done[b] + T, bs)
        sub.block_table.copy_(torch.from_numpy(table[active]).to(torch.int32))
        q = torch.stack([raw_q[b, done[b]:done[b] + T] for b in active]).cuda()
        k = torch.stack([raw_k[b, done[b]:done[b] + T] for b in active]).cuda()
        v = torch.stack([raw_v[b, done[b]:done[b] + T] for b in active]).cuda()
        sk.paged_append(tbl, sub, q, k, v)
        layer.seq_lens[active] = sub.seq_lens
        for i, b in enumerate(active):
            done[b] += T
            q_last[b] = q[i, -1]
            alloc.release_outside(table, b, done[b], bs, S, W, sink_len)
    assert done == list(lengths)
    # freed entries are -1 in the device table too (the kernel must never read them)
    layer.block_table.copy_(torch.from_numpy(table).to(torch.int32))
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    assert layer.seq_lens.tolist() == list(lengths)
    return layer, table, sink_ids, sink_k, sink_v, raw_q, raw_k, raw_v, q_last, spec


def _oracle_pool(layer_shape, table, sink_ids, sink_k, sink_v, raw_k, raw_v, lengths, spec, bs, r):
    """The oracle's own pool: rotated raw keys placed by the same block table."""
    n_blocks, Hkv, _, D = layer_shape
    kp = np.zeros((n_blocks, Hkv, bs, D))
    vp = np.zeros((n_blocks, Hkv, bs, D))
    for j, blk in enumerate(sink_ids):
        kp[blk] = f64(sink_k[j])
        vp[blk] = f64(sink_v[j])
    for b, L in enumerate(lengths):
        kr = rope_rotate(f64(raw_k[b, :L]), np.arange(L), spec.omega(), 1.0, r, spec.neox)
        for P in range(L):
            blk = table[b, P // bs]
            if blk >= 0:
                kp[blk, :, P % bs] = kr[P]
                vp[blk, :, P % bs] = f64(raw_v[b, P])
    return kp, vp


CASES = [
    # dtype, D, r, Hq, Hkv, bs, S, W, static sink blocks, lengths, chunks
    (torch.bfloat16, 128, 128, 8, 2, 16, 4, 100, 0, [1, 15, 16, 17, 250, 700], [1, 14, 1, 1, 200, 33, 450]),
    (torch.bfloat16, 128, 64, 8, 2, 16, 16, 64, 1, [5, 80, 333], [5, 75, 253]),
    (torch.float32, 64, 64, 4, 2, 8, 2, 37, 0, [3, 90, 301], [3, 87, 211]),
    (torch.bfloat16, 128, 128, 4, 4, 32, 0, 0, 0, [40, 129, 300], [40, 89, 171]),      # full attention
    (torch.bfloat16, 128, 128, 8, 2, 4, 4, 50, 2, [7, 200], [7, 193]),                # 4-token blocks
    # blocks as tall as the kernel's tile and taller: tiles start at key multiples of the
    # tile height inside a block, the window starts anywhere
    (torch.bfloat16, 128, 128, 8, 2, 64, 4, 130, 1, [64, 65, 500], [64, 1, 435]),
    (torch.bfloat16, 128, 128, 8, 2, 128, 4, 301, 0, [300, 777, 1025], [300, 477, 248]),
    (torch.bfloat16, 128, 64, 4, 1, 256, 2, 517, 1, [513, 1100], [513, 587]),
]


# GPT-J (interleaved) pairing through the paged append: partial and full rotary, bf16
# and fp32, with and without static sink blocks
GPTJ_CASES = [CASES[1], CASES[2], CASES[0], CASES[5]]


@pytest.mark.parametrize("case,neox", [(c, True) for c in CASES] + [(c, False) for c in GPTJ_CASES],
                         ids=[f"case{i}" for i in range(len(CASES))] +
                             [f"gptj{i}" for i in range(len(GPTJ_CASES))])
def test_paged_append_and_decode_match_oracle(sk, case, neox):
    dtype, D, r, Hq, Hkv, bs, S, W, nsb, lengths, chunks = case
    layer, table, sink_ids, sink_k, sink_v, raw_q, raw_k, raw_v, q_last, spec = _run_paged(
        sk, dtype=dtype, D=D, r=r, Hq=Hq, Hkv=Hkv, bs=bs, S=S, W=W, n_sink_blocks=nsb, lengths=lengths,
        chunks=chunks, seed=300, neox=neox)
    kp, vp = _oracle_pool(tuple(layer.k_pool.shape), table, sink_ids, sink_k, sink_v, raw_k, raw_v, lengths, spec,
                          bs, r)
    sink_len = nsb * bs
    # the pool rows the append wrote: every kept request row against the oracle's rotation
    for b, L in enumerate(lengths):
        for P in range(L):
            blk = table[b, P // bs]
            if blk < 0:
                continue
            assert_rows_close(f64(layer.k_pool[blk, :, P % bs]), kp[blk, :, P % bs], dtype)
            assert np.array_equal(f64(layer.v_pool[blk, :, P % bs]), vp[blk, :, P % bs])
    out = f64(sk.paged_decode_attention(layer, q_last))
    tol = F32_ATTN_ATOL if dtype == torch.float32 else BF16_ATTN_ATOL
    for b, L in enumerate(lengths):
        full_row = np.concatenate([np.array(sink_ids, dtype=np.int64), table[b]])
        qr = rope_rotate(f64(raw_q[b, L - 1:L]), [L - 1], spec.omega(), 1.0, r, neox)[0]
        want = paged_decode_attention(qr, kp, vp, full_row, L + sink_len, bs, S, W if W > 0 else None)
        np.testing.assert_allclose(out[b], want, rtol=0, atol=tol)
    assert layer.error_bits() == 0


def test_paged_empty_request_and_learned_sinks(sk):
    """A request with no tokens gets zeros; learned sink logits work on paged layers."""
    from sink_kv_attention_gb300 import synth
    layer, table, sink_ids, sink_k, sink_v, raw_q, raw_k, raw_v, q_last, spec = _run_paged(
        sk, dtype=torch.bfloat16, D=128, r=128, Hq=8, Hkv=2, bs=16, S=4, W=60, n_sink_blocks=0,
        lengths=[90, 130], chunks=[90, 40], seed=310)
    kp, vp = _oracle_pool(tuple(layer.k_pool.shape), table, sink_ids, sink_k, sink_v, raw_k, raw_v, [90, 130], spec,
                          16, 128)
    z = torch.linspace(-12.0, 16.0, 8)
    out = f64(sk.paged_decode_attention(layer, q_last, sink_logits=z.cuda()))
    for b, L in enumerate([90, 130]):
        qr = rope_rotate(f64(raw_q[b, L - 1:L]), [L - 1], spec.omega(), 1.0, 128)[0]
        want = paged_decode_attention(qr, kp, vp, table[b], L, 16, 4, 60, sink_logits=z.numpy())
        np.testing.assert_allclose(out[b], want, rtol=0, atol=BF16_ATTN_ATOL)
    layer.seq_lens[0] = 0
    out = sk.paged_decode_attention(layer, q_last)
    assert not out[0].float().abs().any()


def test_paged_window_decode_full_size_sampled(sk):
    """The windowed decode step's shapes on a paged cache: B=32, H_q=32, H_kv=8,
    d_h=128, request sinks S=4, W=4092, 16-token blocks scattered over the pool, only
    the sink block and the window's blocks allocated; 6 requests checked."""
    from sink_kv_attention_gb300 import synth
    c = synth.WINDOW
    B, Hq, Hkv, D, S, W, bs = c["B"], c["Hq"], c["Hkv"], c["D"], c["S"], c["W"], 16
    pos = synth.randint((B,), 13, c["pos_lo"], c["pos_hi"] + 1).tolist()
    max_blocks = blocks_for_tokens(max(pos), bs)
    per_req = 1 + window_span(W, bs)
    n_blocks = B * per_req + 4
    layer = sk.PagedLayer.allocate(B, Hkv, D, block_size=bs, n_blocks=n_blocks, max_blocks=max_blocks,
                                   sinks=S, window=W)
    synth.fill_normal_(layer.k_pool, 11)
    synth.fill_normal_(layer.v_pool, 12)
    rng = np.random.default_rng(14)
    perm = rng.permutation(n_blocks)
    table = np.full((B, max_blocks), -1, dtype=np.int64)
    nxt = 0
    for b in range(B):
        L = pos[b]
        vis = visible_positions(L - 1, S + W, S)
        for j in sorted({k // bs for k in vis}):
            table[b, j] = perm[nxt]
            nxt += 1
    layer.block_table.copy_(torch.from_numpy(table).to(torch.int32))
    layer.seq_lens.copy_(torch.tensor(pos))
    q = synth.normal((B, Hq, D), 15, torch.bfloat16).cuda()
    out = f64(sk.paged_decode_attention(layer, q))
    for b in [0, 3, 9, 17, 26, 31]:
        # the request's blocks (inputs written by the test), compacted for the oracle
        used = [int(x) for x in table[b] if x >= 0]
        idx = torch.tensor(used, device="cuda")
        kp, vp = f64(layer.k_pool[idx]), f64(layer.v_pool[idx])
        row = np.array([used.index(int(x)) if x >= 0 else -1 for x in table[b]])
        want = paged_decode_attention(f64(q[b]), kp, vp, row, pos[b], bs, S, W)
        np.testing.assert_allclose(out[b], want, rtol=0, atol=BF16_ATTN_ATOL)
    assert layer.error_bits() == 0


def window_span(W, bs):
    """Blocks a window of W keys can touch (the oracle's window_blocks with W + 1 keys
    behind, as the visible window here includes the query)."""
    return blocks_for_tokens(W - 1, bs) + 1


def test_paged_errors_are_reported(sk):
    from sink_kv_attention_gb300 import synth
    D, bs = 128, 16
    tbl = sk.RopeTable(D, D, 1e4, 256)
    layer = sk.PagedLayer.allocate(1, 1, D, block_size=bs, n_blocks=4, max_blocks=2, sinks=0, window=0)
    layer.block_table.copy_(torch.tensor([[2, -1]], dtype=torch.int32))
    k = synth.normal((1, 16, 1, D), 1, torch.bfloat16).cuda()
    sk.paged_append(tbl, layer, None, k.clone(), k.clone())
    torch.cuda.synchronize()
    assert layer.error_bits() == 0 and int(layer.seq_lens[0]) == 16
    # the next block is missing (-1): the token is not stored, the error word says so
    sk.paged_append(tbl, layer, None, k[:, :1].clone(), k[:, :1].clone())
    assert layer.error_bits() & sk.SK_DEVERR_BLOCK_TABLE
    layer.err.zero_()
    # past max_blocks * block_size: the request is skipped
    before = int(layer.seq_lens[0])
    sk.paged_append(tbl, layer, None, k.clone(), k.clone())
    assert layer.error_bits() & sk.SK_DEVERR_CAPACITY and int(layer.seq_lens[0]) == before
    layer.err.zero_()
    # decode over a table entry outside the pool: reported, block 0 read instead
    layer.block_table.copy_(torch.tensor([[7, 1]], dtype=torch.int32))
    layer.seq_lens.fill_(16)
    q = synth.normal((1, 1, D), 2, torch.bfloat16).cuda()
    out = sk.paged_decode_attention(layer, q)
    torch.cuda.synchronize()
    assert layer.error_bits() & sk.SK_DEVERR_BLOCK_TABLE
    assert torch.isfinite(out.float()).all()
