"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and lays out buffers; it holds none of the
method's arithmetic (no rotation, no ring rule, no attention).  Tests feed the same
draws to the CUDA path and to the float64 oracle; the benchmark uses them too.

Workloads (names used across tests and the benchmark):
  tiny        1 sequence, 1 layer, H_q=8, H_kv=4, d_h=r=64, theta=1e4, fp32 N(0,1),
              C=6 with S=2 sinks, 10 tokens decoded one at a time
  window      windowed-layer decode step: B=32, H_q=32, H_kv=8, d_h=r=128,
              theta=5e5, bf16 N(0,1), S=4 + W=4092 (C=4096), positions U[4096, 32768],
              ring full with a random head
  hybrid      Llama-3-8B-shaped decode: 32 layers, layer i global iff (i+1) % 4 == 0,
              B=16, H_q=32, H_kv=8, d_h=128, bf16, sliding S=4 + W=4096, global
              layers holding a 131072-token prefix
  prefill     B=1, T=32768, H_q=32, H_kv=8, d_h=r=128, bf16 N(0,1), S=4, W=4092
  rerotate    1 sequence, 48 layers, H_kv=4, d_h=128, r=64, 524288 cached positions,
              K ~ U(-1, 1), YaRN factor 1 -> 2 with L0=262144
"""
from __future__ import annotations

import torch


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, dtype=torch.float32, device="cpu") -> torch.Tensor:
    """N(0, 1) draws in float32, then cast (bf16 inputs are the rounded draws)."""
    g = generator(seed, device)
    return torch.randn(*shape, generator=g, dtype=torch.float32, device=device).to(dtype)


def uniform(shape, seed: int, lo: float, hi: float, dtype=torch.float32, device="cpu") -> torch.Tensor:
    g = generator(seed, device)
    x = torch.rand(*shape, generator=g, dtype=torch.float32, device=device)
    return (x * (hi - lo) + lo).to(dtype)


def randint(shape, seed: int, lo: int, hi: int, device="cpu") -> torch.Tensor:
    """Integers uniform in [lo, hi)."""
    g = generator(seed, device)
    return torch.randint(lo, hi, tuple(shape), generator=g, dtype=torch.int64, device=device)


def sparse_signs(shape, seed: int, density: float, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """Values in {-1, 0, +1}: each entry is +1 or -1 with probability density / 2 each,
    else 0.  Exact in every float format; sums of them are small integers."""
    g = generator(seed, device)
    u = torch.rand(*shape, generator=g, dtype=torch.float32, device=device)
    x = torch.zeros_like(u)
    x[u < density / 2] = 1.0
    x[(u >= density / 2) & (u < density)] = -1.0
    return x.to(dtype)


def fill_sparse_signs_(t: torch.Tensor, seed: int, density: float) -> torch.Tensor:
    """sparse_signs into a (possibly huge) device tensor, in place."""
    g = generator(seed, t.device)
    flat = t.view(-1)
    step = 1 << 28
    for i in range(0, flat.numel(), step):
        chunk = flat[i:i + step]
        u = torch.rand(chunk.numel(), generator=g, dtype=torch.float32, device=t.device)
        chunk.copy_(torch.where(u < density / 2, 1.0, torch.where(u < density, -1.0, 0.0)))
    return t


def fill_normal_(t: torch.Tensor, seed: int) -> torch.Tensor:
    """Fill a (possibly huge) device tensor with N(0,1) draws, in place."""
    g = generator(seed, t.device)
    flat = t.view(-1)
    step = 1 << 28
    for i in range(0, flat.numel(), step):
        chunk = flat[i:i + step]
        chunk.copy_(torch.randn(chunk.numel(), generator=g, dtype=torch.float32, device=t.device))
    return t


def fill_uniform_(t: torch.Tensor, seed: int, lo: float, hi: float) -> torch.Tensor:
    g = generator(seed, t.device)
    flat = t.view(-1)
    step = 1 << 28
    for i in range(0, flat.numel(), step):
        chunk = flat[i:i + step]
        r = torch.rand(chunk.numel(), generator=g, dtype=torch.float32, device=t.device)
        chunk.copy_(r * (hi - lo) + lo)
    return t


# Shapes of the workloads (see the module docstring).
TINY = dict(B=1, Hq=8, Hkv=4, D=64, r=64, theta=1e4, S=2, W=4, T=10)
WINDOW = dict(B=32, Hq=32, Hkv=8, D=128, r=128, theta=5e5, S=4, W=4092, pos_lo=4096, pos_hi=32768)
HYBRID = dict(layers=32, B=16, Hq=32, Hkv=8, D=128, r=128, theta=5e5, S=4, W=4096, prefix=131072)
PREFILL = dict(B=1, T=32768, Hq=32, Hkv=8, D=128, r=128, theta=5e5, S=4, W=4092)
REROTATE = dict(layers=48, B=1, Hkv=4, D=128, r=64, theta=5e5, positions=524288, orig_ctx=262144,
                factor_a=1.0, factor_b=2.0)


def hybrid_layer_is_global(i: int) -> bool:
    """Layer assignment of the 3:1 sliding:global pattern (layer i global iff (i+1) % 4 == 0)."""
    return (i + 1) % 4 == 0


def window_state(seed: int, B: int, W: int, pos_lo: int, pos_hi: int):
    """Ring state of the windowed decode workload before its step: tokens seen per
    sequence U[pos_lo, pos_hi], ring full (count = W) with a head U[0, W)."""
    pos = randint((B,), seed, pos_lo, pos_hi + 1)
    head = randint((B,), seed + 1, 0, W).to(torch.int32)
    count = torch.full((B,), W, dtype=torch.int32)
    return pos, head, count
