"""Float64 CPU oracle for sink + window KV attention with RoPE / YaRN.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference leg may import this module.  The CUDA
library (``sink_kv_attention_gb300``) never imports it, and this module imports
nothing from the library: the two share no code.

Everything here is a plain, slow restatement of what the source pages compute,
in float64 numpy, one function per step, each citing the passage it follows.
Page names used in the citations:

* "RoPE, scaling, sliding window, attention sinks" (mlinterviewnotes, page 1)
* "Inference & 128K Long Context" / "KV-Cache Engineering" (GPT-OSS-Lite, page 2)
* "#2961 rope: --rope-scaling dynamic" (strata pull request, page 3)
* "Attention Sink 与 Streaming KV Cache" (llm-glossary, page 4)

Precision: float64 throughout, including where a floating-point value decides an
integer (the int8 code rint(x / scale) of ``quantize_int8_rows``).  Parity tests
treat values within 1e-3 of a rounding tie as undecided: there either neighbour
is a correct rounding.

Parity status: every function below is pinned by ``tests/test_oracle_*.py``
against values the pages print, closed forms, invariants or library routines.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np


# ---------------------------------------------------------------------------
# O1. Rotary frequencies: plain RoPE and the YaRN blend.
# ---------------------------------------------------------------------------

def rope_inv_freq(rotary_dim: int, theta: float) -> np.ndarray:
    """omega_i = theta ** (-2 i / r) for the r/2 rotary pairs i = 0 .. r/2-1.

    "RoPE, scaling, sliding window, attention sinks", section on RoPE: the
    ``_compute_inv_freq`` listing, 1 / base ** (arange(0, r, 2) / r).
    """
    i = np.arange(rotary_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / rotary_dim)


def yarn_correction_dim(num_rotations: float, rotary_dim: int, theta: float,
                        orig_ctx: int) -> float:
    """Pair index at which a pair turns ``num_rotations`` times in ``orig_ctx`` tokens.

    "RoPE, scaling, sliding window, attention sinks", "YaRN, precisely":
    d(n) = r * ln(L0 / (2 pi n)) / (2 ln b).
    """
    return (rotary_dim * math.log(orig_ctx / (num_rotations * 2.0 * math.pi))
            / (2.0 * math.log(theta)))


def yarn_correction_range(beta_fast: float, beta_slow: float, rotary_dim: int,
                          theta: float, orig_ctx: int):
    """(low, high) = (floor d(beta_fast), ceil d(beta_slow)), clamped to [0, r-1].

    "RoPE, scaling, sliding window, attention sinks", "YaRN, precisely" (the worked
    band "truncated to [20, 46]") and its first exercise (max(lo, 0), min(hi, r-1)).
    """
    low = math.floor(yarn_correction_dim(beta_fast, rotary_dim, theta, orig_ctx))
    high = math.ceil(yarn_correction_dim(beta_slow, rotary_dim, theta, orig_ctx))
    return max(low, 0), min(high, rotary_dim - 1)


def yarn_linear_ramp(low: float, high: float, n: int) -> np.ndarray:
    """clamp((i - low) / (high - low), 0, 1) for i < n; high += 0.001 when low == high.

    "RoPE, scaling, sliding window, attention sinks", "YaRN, precisely"
    (``yarn_linear_ramp_mask``).
    """
    if low == high:
        high = high + 0.001
    i = np.arange(n, dtype=np.float64)
    return np.clip((i - low) / (high - low), 0.0, 1.0)


def yarn_mscale(factor: float) -> float:
    """mu = 1 for s <= 1, else 0.1 ln s + 1.

    "RoPE, scaling, sliding window, attention sinks", "YaRN, precisely"
    (``yarn_get_mscale``; mu(8) = 1.2079).
    """
    if factor <= 1.0:
        return 1.0
    return 0.1 * math.log(factor) + 1.0


def yarn_inv_freq(rotary_dim: int, theta: float, factor: float, orig_ctx: int,
                  beta_fast: float = 32.0, beta_slow: float = 1.0) -> np.ndarray:
    """YaRN frequencies: blend of the extrapolated and the interpolated sets.

    "RoPE, scaling, sliding window, attention sinks", "YaRN, precisely": with
    pos_freq_i = b ** (2i / r), extrapolation = 1 / pos_freq, interpolation =
    1 / (s pos_freq), mask = (1 - ramp) * extrapolation_factor (= 1), and
    omega = interpolation * (1 - mask) + extrapolation * mask.
    """
    pos_freq = np.power(float(theta),
                        np.arange(0, rotary_dim, 2, dtype=np.float64) / rotary_dim)
    extrapolation = 1.0 / pos_freq
    interpolation = 1.0 / (factor * pos_freq)
    low, high = yarn_correction_range(beta_fast, beta_slow, rotary_dim, theta, orig_ctx)
    mask = 1.0 - yarn_linear_ramp(low, high, rotary_dim // 2)
    return interpolation * (1.0 - mask) + extrapolation * mask


@dataclass(frozen=True)
class RopeSpec:
    """The rotary configuration: head_dim d_h, rotary_dim r <= d_h, base theta,
    NeoX or GPT-J pairing, optional YaRN factor (<= 1 means plain RoPE)."""
    head_dim: int
    rotary_dim: int
    theta: float
    neox: bool = True
    yarn_factor: float = 1.0
    yarn_orig_ctx: int = 4096
    beta_fast: float = 32.0
    beta_slow: float = 1.0

    def omega(self) -> np.ndarray:
        """Plain frequencies when the factor is <= 1 ("none"), else the YaRN blend."""
        if self.yarn_factor <= 1.0:
            return rope_inv_freq(self.rotary_dim, self.theta)
        return yarn_inv_freq(self.rotary_dim, self.theta, self.yarn_factor,
                             self.yarn_orig_ctx, self.beta_fast, self.beta_slow)

    def mscale(self) -> float:
        return yarn_mscale(self.yarn_factor)

    def with_factor(self, factor: float) -> "RopeSpec":
        return RopeSpec(self.head_dim, self.rotary_dim, self.theta, self.neox, factor,
                        self.yarn_orig_ctx, self.beta_fast, self.beta_slow)


# ---------------------------------------------------------------------------
# O2. Rotation of Q or K (never V).
# ---------------------------------------------------------------------------

def rotary_pairs(rotary_dim: int, neox: bool):
    """Indices (first, second) of each rotary pair.

    "RoPE, scaling, sliding window, attention sinks", section on RoPE: NeoX pairs
    element j with j + r/2, GPT-J pairs 2j with 2j+1.
    """
    half = rotary_dim // 2
    if neox:
        return np.arange(half), np.arange(half) + half
    return np.arange(0, rotary_dim, 2), np.arange(1, rotary_dim, 2)


def rope_rotate(x: np.ndarray, positions: Sequence[int], omega: np.ndarray,
                mscale: float, rotary_dim: int, neox: bool = True) -> np.ndarray:
    """Rotate each rotary pair of x by angle P * omega_j and scale it by mscale.

    x has shape [n_tok, H, D] (any H), positions has n_tok entries.  For pair j
    with elements (x1, x2) and angle a = P omega_j:
        o1 = mscale (x1 cos a - x2 sin a),  o2 = mscale (x2 cos a + x1 sin a);
    dims [r, D) pass through unchanged.

    "RoPE, scaling, sliding window, attention sinks": the rotation listing
    (o1 = x1 cos - x2 sin, o2 = x2 cos + x1 sin), partial rotary (the tail passes
    through) and the YaRN table whose cos and sin both carry mscale.
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    first, second = rotary_pairs(rotary_dim, neox)
    pos = np.asarray(positions, dtype=np.float64).reshape(-1, 1)
    angle = pos * np.asarray(omega, dtype=np.float64).reshape(1, -1)     # [n_tok, r/2]
    c = (np.cos(angle) * mscale)[:, None, :]
    s = (np.sin(angle) * mscale)[:, None, :]
    x1 = x[..., first]
    x2 = x[..., second]
    out[..., first] = x1 * c - x2 * s
    out[..., second] = x2 * c + x1 * s
    return out


def rope_table(spec: RopeSpec, n_positions: int) -> np.ndarray:
    """The cos/sin table for positions 0 .. n_positions-1: [n_positions, r/2, 2] with
    entry (P, j) = mscale (cos(P omega_j), sin(P omega_j)), in float64.

    "RoPE, scaling, sliding window, attention sinks": the rotation gathers rows of a
    table built once per configuration ("Hybrid models break the uniform-spec
    assumption", the walk of one decode token), and YaRN's mscale rides on both cos
    and sin ("YaRN, precisely").
    """
    angle = np.arange(n_positions, dtype=np.float64)[:, None] * spec.omega()[None, :]
    mu = spec.mscale()
    return np.stack([mu * np.cos(angle), mu * np.sin(angle)], axis=-1)


def rerotate(k_a: np.ndarray, positions: Sequence[int], spec_a: RopeSpec,
             spec_b: RopeSpec) -> np.ndarray:
    """Turn keys stored rotated under spec A into keys rotated under spec B.

    "#2961 rope: --rope-scaling dynamic", "What it does": since keys are cached after
    RoPE, each pair is turned by a further angle p * (w_B - w_A) and scaled by
    mscale_B / mscale_A; this is R_a R_b = R_{a+b} ("Attention Sink 与 Streaming KV Cache", RoPE section).
    No raw key is needed.
    """
    delta = spec_b.omega() - spec_a.omega()
    return rope_rotate(k_a, positions, delta, spec_b.mscale() / spec_a.mscale(),
                       spec_a.rotary_dim, spec_a.neox)


# ---------------------------------------------------------------------------
# int8 keys with one scale per row.
# ---------------------------------------------------------------------------

def quantize_int8_rows(x: np.ndarray):
    """Symmetric absmax int8 codes with one scale per row (last axis), in float64.

    scale = max_k |x_k| / 127 (a zero row gets scale 1 and codes 0);
    code = clamp(rint(x / scale), -127, 127), rint rounding half to even.
    "#2961 rope: --rope-scaling dynamic", "What it does": int8 keys are dequantized,
    turned and requantized; its parity table measures errors in int8 steps (the
    scale).  The pages fix neither the scale rule nor the rounding; the reading
    taken is the symmetric absmax rule with one scale per row, its division and
    rounding done on the float64 row as written here.
    """
    x = np.asarray(x, dtype=np.float64)
    amax = np.max(np.abs(x), axis=-1, keepdims=True)
    zero = amax == 0.0
    scale = np.where(zero, 1.0, amax / 127.0)
    q = np.where(zero, 0.0, np.rint(x / scale))
    codes = np.clip(q, -127, 127).astype(np.int8)
    return codes, scale[..., 0]


def dequantize_int8_rows(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """x = code * scale in float64."""
    return codes.astype(np.float64) * np.asarray(scale, dtype=np.float64)[..., None]


def rerotate_int8(codes: np.ndarray, scale: np.ndarray, positions: Sequence[int],
                  spec_a: RopeSpec, spec_b: RopeSpec):
    """Dequantize, turn the rotary pairs (``rerotate``), requantize with a new scale.

    "#2961 rope: --rope-scaling dynamic", "What it does" (int8 K without the
    Hadamard: dequantize, turn the rotary pairs, requantize).  One scale per row
    over all D dims, so the tail codes may change on requantisation.
    codes: [n_tok, H, D] int8, scale: [n_tok, H].
    """
    x = dequantize_int8_rows(codes, scale)
    turned = rerotate(x, positions, spec_a, spec_b)
    new_codes, new_scale = quantize_int8_rows(turned)
    return new_codes, new_scale, turned


# ---------------------------------------------------------------------------
# O4. Per-layer caches: ring with pinned sinks, and the global linear prefix.
# ---------------------------------------------------------------------------

class CapacityError(RuntimeError):
    """A global-layer append past its capacity: a loud error, never a truncation
    ("KV-Cache Engineering", 4.6 and 6: hitting the context cap fails loudly)."""


class RingCache:
    """One (sequence, layer) windowed cache: S pinned sink slots then a ring of W.

    The ring follows "Inference & 128K Long Context", "MixedKVCache", windowed
    layers (write at head, head = (head+1) % W, count = min(W, count+1); a chunk of
    n >= W keeps its last W rows with head = 0, count = W), extended with S sink
    slots that hold positions 0..S-1 and are never overwritten ("Attention Sink 与
    Streaming KV Cache": sink + recent).  ``rows`` holds whatever per-token rows the
    caller stores (K, V, ...); ``slot_pos`` records the logical position per slot.
    """

    def __init__(self, sinks: int, window: int):
        assert sinks >= 0 and window >= 1
        self.S = sinks
        self.W = window
        self.C = sinks + window
        self.slots: List[object] = [None] * self.C
        self.slot_pos = [-1] * self.C
        self.pos = 0      # tokens seen = the next absolute position
        self.head = 0     # next ring index to write, in [0, W)
        self.count = 0    # valid ring entries, in [0, W]

    def append(self, rows: Sequence[object]) -> None:
        T = len(rows)
        ring_items = []
        for t in range(T):
            P = self.pos + t
            if P < self.S:
                self.slots[P] = rows[t]
                self.slot_pos[P] = P
            else:
                ring_items.append((P, rows[t]))
        n = len(ring_items)
        if n >= self.W:
            for j, (P, row) in enumerate(ring_items[n - self.W:]):
                self.slots[self.S + j] = row
                self.slot_pos[self.S + j] = P
            self.head = 0
            self.count = self.W
        else:
            for t, (P, row) in enumerate(ring_items):
                j = (self.head + t) % self.W
                self.slots[self.S + j] = row
                self.slot_pos[self.S + j] = P
            self.head = (self.head + n) % self.W
            self.count = min(self.W, self.count + n)
        self.pos += T

    def chronological_slots(self) -> List[int]:
        """Slots in temporal order: the sinks, then ring[head:] + ring[:head] when
        the ring is full, else ring[:count] ("Inference & 128K Long Context",
        "MixedKVCache", read ordering)."""
        sinks = list(range(min(self.pos, self.S)))
        if self.count == self.W:
            ring = list(range(self.head, self.W)) + list(range(0, self.head))
        else:
            ring = list(range(self.count))
        return sinks + [self.S + j for j in ring]

    def chronological_positions(self) -> List[int]:
        return [self.slot_pos[s] for s in self.chronological_slots()]

    def chronological_rows(self) -> List[object]:
        return [self.slots[s] for s in self.chronological_slots()]


class GlobalCache:
    """A global layer's linear prefix: rows [0, len), an append writes at len and
    advances it; past ``capacity`` it raises ("KV-Cache Engineering", 4.6 and 5.2,
    global branch; the growth policy itself belongs to the host allocator)."""

    def __init__(self, capacity: int):
        self.capacity = capacity
        self.rows: List[object] = []

    @property
    def pos(self) -> int:
        return len(self.rows)

    def append(self, rows: Sequence[object]) -> None:
        if len(self.rows) + len(rows) > self.capacity:
            raise CapacityError(f"global layer: {len(self.rows)} + {len(rows)} > "
                                f"capacity {self.capacity}")
        self.rows.extend(rows)

    def chronological_positions(self) -> List[int]:
        return list(range(len(self.rows)))

    def chronological_rows(self) -> List[object]:
        return list(self.rows)


def shift_recent_keys(cache: "RingCache", delta: int, omega: np.ndarray, rotary_dim: int,
                      neox: bool = True) -> None:
    """Turn every occupied recent (ring) key of ``cache`` by ``delta`` positions, in
    place; sink keys and all values stay as they are.

    "Attention Sink 与 Streaming KV Cache", "RoPE：absolute positions 与 local
    rerotation 是两种实现": a cache that feeds attention local positions in [0, C-1]
    moves each recent key from local position p to p - 1 when the window slides; a
    key cached as R_p k becomes R_{p+delta} k by one more turn of delta positions
    (R_a R_b = R_{a+b}, no raw key needed), with no mscale change, and the sink keys
    keep their local positions.  Rows are (k_rot [H_kv, D], v) pairs.
    """
    for j in range(cache.count):
        s = cache.S + j
        k, v = cache.slots[s]
        turned = rope_rotate(np.asarray(k)[None], [delta], omega, 1.0, rotary_dim, neox)[0]
        cache.slots[s] = (turned, v)


# ---------------------------------------------------------------------------
# O5. The visible set of a query.
# ---------------------------------------------------------------------------

def visible_positions(P: int, capacity: int, sinks: int) -> List[int]:
    """V(P) for capacity C, sinks S < C, recent W = C - S: all of 0..P when P < C,
    else 0..S-1 together with max(S, P-W+1)..P.

    "Attention Sink 与 Streaming KV Cache", "可见集合与容量定义" and the C=6, S=2,
    T=10 worked example.
    """
    if P < capacity:
        return list(range(P + 1))
    recent = capacity - sinks
    start = max(sinks, P - recent + 1)
    return list(range(sinks)) + list(range(start, P + 1))


def mask_allows(P: int, k: int, sinks: int, window: Optional[int]) -> bool:
    """Mask rule for a query at absolute position P and a key at absolute k:
    causal (k <= P) and either a sink (k < S) or recent (P - k < W).  window None
    means a global layer (causal only).

    "KV-Cache Engineering", 5.5: keys allowed where idx_q >= idx_k and
    idx_q - idx_k < window; with sinks added as in "Attention Sink 与 Streaming KV
    Cache" (sink ∪ recent).
    """
    if k > P:
        return False
    if window is None:
        return True
    return k < sinks or (P - k) < window


# ---------------------------------------------------------------------------
# O6. Attention.
# ---------------------------------------------------------------------------

# Bounds of a learned sink logit ("Inference & 128K Long Context", "Sink clamp cache":
# the forward pass clamps the trained per-head sink bias to [-10, 15]).
SINK_LOGIT_MIN = -10.0
SINK_LOGIT_MAX = 15.0


def clamp_sink_logits(sink_logits) -> np.ndarray:
    """The per-head learned sink logits as the forward pass uses them: clamped to
    [SINK_LOGIT_MIN, SINK_LOGIT_MAX] ("Inference & 128K Long Context", "Sink clamp
    cache")."""
    return np.clip(np.asarray(sink_logits, dtype=np.float64), SINK_LOGIT_MIN, SINK_LOGIT_MAX)


def attend(q: np.ndarray, keys: np.ndarray, values: np.ndarray,
           sink_logits: Optional[Sequence[float]] = None) -> np.ndarray:
    """Softmax attention of one query row over a key/value set, with GQA.

    q [H_q, D], keys and values [n, H_kv, D]; q head h reads kv head h // n_rep
    ("KV-Cache Engineering", 5.5, ``repeat_kv``).  scores = q . k / sqrt(D), a
    max-subtracted softmax in float64, out = sum_j p_j v_j ("Attention Sink 与
    Streaming KV Cache", the experiment's ``incremental_sink``).

    ``sink_logits`` ([H_q], optional): learned sinks, a trained per-head scalar whose
    exponential joins the softmax denominator and that carries no value
    ("RoPE, scaling, sliding window, attention sinks", "Hybrid models break the
    uniform-spec assumption", the second kind of sink; clamped as
    ``clamp_sink_logits``).  Reading: the scalar is a logit in
    the units of the scaled scores, so head h's weights are
    exp(s_j) / (sum_i exp(s_i) + exp(z_h)).
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    Hq, D = q.shape
    Hkv = keys.shape[1]
    n_rep = Hq // Hkv
    z = None if sink_logits is None else clamp_sink_logits(sink_logits)
    out = np.zeros((Hq, D), dtype=np.float64)
    for h in range(Hq):
        g = h // n_rep
        s = keys[:, g, :] @ q[h] / math.sqrt(D)
        if z is None:
            s = s - s.max()
            p = np.exp(s)
            p = p / p.sum()
        else:
            m = max(s.max(), z[h])
            e = np.exp(s - m)
            p = e / (e.sum() + math.exp(z[h] - m))
        out[h] = p @ values[:, g, :]
    return out


def decode_attention(cache, q_rot: np.ndarray,
                     sink_logits: Optional[Sequence[float]] = None) -> np.ndarray:
    """Decode attention of one new query over a cache after its own append:
    the cache's chronological rows are exactly the visible set V(P).

    Rows of the cache are (k_rot, v) pairs of shape [H_kv, D] each.
    "Inference & 128K Long Context", "_attn_forward_layer" (append, get, attend).
    ``sink_logits``: optional learned per-head sinks, as in ``attend``.
    """
    rows = cache.chronological_rows()
    keys = np.stack([r[0] for r in rows])
    values = np.stack([r[1] for r in rows])
    return attend(q_rot, keys, values, sink_logits)


def prefill_attention(q_rot: np.ndarray, k_rot: np.ndarray, v: np.ndarray, p0: int,
                      sinks: int, window: Optional[int],
                      rows: Optional[Sequence[int]] = None,
                      sink_logits: Optional[Sequence[float]] = None) -> np.ndarray:
    """Masked attention of a prompt chunk over itself.

    q_rot [T, H_q, D], k_rot and v [T, H_kv, D]; chunk index t has absolute
    position p0 + t.  Query t sees key k iff ``mask_allows(p0+t, p0+k, S, W)``.
    ``rows`` picks the query indices to evaluate (all by default).
    ``sink_logits``: optional learned per-head sinks, as in ``attend``.
    Returns [len(rows), H_q, D].
    """
    T = q_rot.shape[0]
    if rows is None:
        rows = range(T)
    out = []
    for t in rows:
        P = p0 + t
        ks = [k for k in range(T) if mask_allows(P, p0 + k, sinks, window)]
        out.append(attend(q_rot[t], k_rot[ks], v[ks], sink_logits))
    return np.stack(out)


def prefill_attention_prior(q_rot: np.ndarray, k_rot: np.ndarray, v: np.ndarray, prior,
                            sinks: int, window: Optional[int],
                            rows: Optional[Sequence[int]] = None,
                            sink_logits: Optional[Sequence[float]] = None) -> np.ndarray:
    """Masked attention of a prompt chunk that continues a cached sequence.

    ``prior`` is the sequence's RingCache or GlobalCache before the chunk (rows are
    (k_rot, v) pairs [H_kv, D]); the chunk starts at p0 = prior.pos.  Query t (position
    P = p0 + t) attends over the keys the cache still holds together with chunk keys
    0..t, keeping those ``mask_allows(P, position, S, W)`` admits.  "KV-Cache
    Engineering", 5.5: the chunk's rotated keys are appended to the cache and the
    queries attend over what the cache returns; the mask places query t at key index
    t + (T_k - T_q), which covers a multi-token chunk over a cached prefix.

    A key that the mask admits but the cache has dropped is an error: the cache must
    have been built with the same sinks and window.
    """
    T = q_rot.shape[0]
    p0 = prior.pos
    cached_pos = list(prior.chronological_positions())
    cached = list(prior.chronological_rows())
    pos_all = cached_pos + [p0 + k for k in range(T)]
    k_all = [np.asarray(r[0], dtype=np.float64) for r in cached] + [k_rot[k] for k in range(T)]
    v_all = [np.asarray(r[1], dtype=np.float64) for r in cached] + [v[k] for k in range(T)]
    have = set(cached_pos)
    if rows is None:
        rows = range(T)
    out = []
    for t in rows:
        P = p0 + t
        for k in range(p0):
            if mask_allows(P, k, sinks, window) and k not in have:
                raise ValueError(f"position {k}, visible from {P}, is not in the prior cache")
        ks = [i for i, pk in enumerate(pos_all) if mask_allows(P, pk, sinks, window)]
        out.append(attend(q_rot[t], np.stack([k_all[i] for i in ks]), np.stack([v_all[i] for i in ks]),
                          sink_logits))
    return np.stack(out)


# ---------------------------------------------------------------------------
# O6b. Paged caches: block tables with static sink blocks.
# ---------------------------------------------------------------------------

def blocks_for_tokens(n_tokens: int, block_size: int) -> int:
    """Blocks holding n tokens: cdiv(n, block_size) ("RoPE, scaling, sliding window,
    attention sinks", the sliding-window section: full attention at 128k and 16-token
    blocks needs cdiv(131072, 16) = 8192 blocks)."""
    return -(-n_tokens // block_size)


def window_blocks(window: int, block_size: int, extra_retained: int = 0, in_flight: int = 0,
                  max_len: Optional[int] = None) -> int:
    """Blocks a sliding-window layer may hold per request: the window's tokens (W - 1
    behind the query, plus retained and in-flight tokens, at most max_len) in whole
    blocks, plus one because the window need not start on a block boundary (same
    section: 257 blocks for W = 4096 and 16-token blocks)."""
    n = window - 1 + extra_retained + in_flight
    if max_len is not None:
        n = min(n, max_len)
    return blocks_for_tokens(n, block_size) + 1


def first_window_token(n_computed: int, window: int, extra_retained: int = 0) -> int:
    """The oldest token a sliding-window query still needs; every block wholly before
    it may be freed (replaced by the null block) (same section, the window edge)."""
    return max(0, n_computed - window + 1 - extra_retained)


def prepend_static_sinks(block_table: np.ndarray, seq_lens: Sequence[int], sink_blocks: Sequence[int],
                         sink_len: int):
    """The attention metadata with static sink blocks ("RoPE, scaling, sliding window,
    attention sinks", "Hybrid models break the uniform-spec assumption", the static
    sink excerpt): the sink blocks go in front of every request's block table and each
    nonzero sequence length grows by sink_len; a length of zero stays zero."""
    n_sink = len(sink_blocks)
    B, nb = block_table.shape
    table = np.zeros((B, n_sink + nb), dtype=np.int64)
    table[:, :n_sink] = np.asarray(sink_blocks)[None, :]
    table[:, n_sink:] = block_table
    lens = np.asarray(seq_lens, dtype=np.int64) + sink_len
    lens[lens == sink_len] = 0
    return table, lens


def paged_logical_rows(k_pool: np.ndarray, v_pool: np.ndarray, table_row: Sequence[int], length: int,
                       block_size: int):
    """The first ``length`` logical (k, v) rows of one request: logical key i lives in
    physical block table_row[i // block_size] at offset i % block_size ("vLLM, from
    the inside out", PagedAttention: blocks, logical blocks, block table).  Pools are
    [n_blocks][H_kv][block_size][D]; returns k and v as [length][H_kv][D]."""
    ks, vs = [], []
    for i in range(length):
        blk = int(table_row[i // block_size])
        ks.append(k_pool[blk, :, i % block_size, :])
        vs.append(v_pool[blk, :, i % block_size, :])
    return np.stack(ks), np.stack(vs)


def paged_decode_attention(q_rot: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                           table_row: Sequence[int], length: int, block_size: int, sinks: int,
                           window: Optional[int],
                           sink_logits: Optional[Sequence[float]] = None) -> np.ndarray:
    """Decode attention of a request's newest query (logical position length - 1) over
    its paged keys: the same visible set as a contiguous cache with capacity
    sinks + window ("Attention Sink 与 Streaming KV Cache", V(P)), every key of a
    full-attention layer (window None) -- only the visible blocks are ever read, so
    freed blocks may hold anything."""
    if length == 0:
        return np.zeros_like(np.asarray(q_rot, dtype=np.float64))
    P = length - 1
    if window is None:
        vis = list(range(length))
    else:
        vis = visible_positions(P, sinks + window, sinks)
    ks, vs = [], []
    for i in vis:
        blk = int(table_row[i // block_size])
        ks.append(k_pool[blk, :, i % block_size, :])
        vs.append(v_pool[blk, :, i % block_size, :])
    return attend(q_rot, np.stack(ks), np.stack(vs), sink_logits)


# ---------------------------------------------------------------------------
# O7. Dynamic factor policy.
# ---------------------------------------------------------------------------

def dynamic_factor(total_positions: int, orig_ctx: int, step: float = 0.125,
                   cap: Optional[float] = None) -> float:
    """1 while the positions fit the trained context; past it, positions / L0
    rounded up to ``step`` and capped.

    "#2961 rope: --rope-scaling dynamic", "What it does", the factor.
    """
    if total_positions <= orig_ctx:
        return 1.0
    f = math.ceil((total_positions / orig_ctx) / step) * step
    if cap is not None:
        f = min(f, cap)
    return f


# ---------------------------------------------------------------------------
# Measurement context.
# ---------------------------------------------------------------------------

def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int,
                       elem_bytes: int) -> int:
    """c = 2 L h_kv d_h bytes ("RoPE, scaling, sliding window, attention sinks",
    sliding-window section: 128 KiB per token for the Llama-3-8B shape)."""
    return 2 * n_layers * n_kv_heads * head_dim * elem_bytes
