"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the tests, the benchmark, the smoke check and the
oracle's callers.  It holds no attention arithmetic: it only draws random
numbers (numpy PCG64, so the same seed gives the same values on any host)
and names the workload shapes.

Workloads (the FlashAttention-3 benchmark protocol sweeps the sequence length
from 512 to 16K with batch chosen so that there are 16K tokens, head
dimension 64/128/256, causal and non-causal -- "FlashAttention-3: async
pipelines on Hopper", section "how to read the paper's performance numbers";
the FP8 error study uses a synthetic distribution with a few large outliers,
section "why FP8 numeric tests must match the model's distribution"):

* tiny   B=1,  H=2,  N=128,   d=64,  N(0,1), seed 0, scale 1/8
* mid    B=4,  H=16, N=2048,  d=128, N(0,1), seed 1
* sweep  N in {512..16384}, B=16384/N, (H,d) in {(32,64),(16,128),(8,256)}, seed 2+idx
* fp8    B=16384/N, H=16, N in {1k,4k,16k}, d=128, fp32 N(0,1) +
         Bernoulli(0.001) * N(0, sigma^2) outliers (sigma = 10), seed 3; Hadamard
         sign seed 4
* long   B=1, H=16, N=65536, d=128, N(0,1), seed 5, causal
"""
from __future__ import annotations

import math

import numpy as np

SWEEP_N = (512, 1024, 2048, 4096, 8192, 16384)
SWEEP_HD = ((32, 64), (16, 128), (8, 256))
TOTAL_TOKENS = 16384
FP8_N = (1024, 4096, 16384)


def normal(shape, seed: int, stream: int = 0) -> np.ndarray:
    """i.i.d. N(0,1) fp32.  ``stream`` separates Q/K/V drawn from one seed."""
    rng = np.random.Generator(np.random.PCG64([seed, stream]))
    return rng.standard_normal(size=shape, dtype=np.float32)


def qkv_normal(shape, seed: int):
    """Q, K, V as three independent N(0,1) fp32 arrays of ``shape``."""
    return normal(shape, seed, 0), normal(shape, seed, 1), normal(shape, seed, 2)


def outliers(shape, seed: int, stream: int = 0, p: float = 1e-3, sigma: float = 10.0) -> np.ndarray:
    """fp32 N(0,1) + Bernoulli(p) * N(0, sigma^2), element-wise independent."""
    rng = np.random.Generator(np.random.PCG64([seed, 100 + stream]))
    base = rng.standard_normal(size=shape, dtype=np.float32)
    hit = rng.random(size=shape, dtype=np.float32) < p
    big = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(sigma)
    return (base + np.where(hit, big, np.float32(0.0))).astype(np.float32)


def qkv_outliers(shape, seed: int = 3, sigma: float = 10.0):
    return tuple(outliers(shape, seed, s, sigma=sigma) for s in range(3))


def hadamard_signs(d: int, seed: int = 4) -> np.ndarray:
    """d random +-1 entries (int8): the random diagonal of the rotation."""
    rng = np.random.Generator(np.random.PCG64([seed, 200]))
    return np.where(rng.random(d) < 0.5, -1, 1).astype(np.int8)


def rope_tables(N: int, d: int, base: float = 10000.0, offset: int = 0):
    """Rotary-embedding angle tables, inputs of the quantiser: (cos, sin),
    fp32 [N, d/2], for positions offset..offset+N-1 and frequencies
    base^(-2i/d), i < d/2 (the usual choice; the pages fix none).  The
    angles are formed in fp64 and rounded once."""
    pos = np.arange(offset, offset + N, dtype=np.float64)[:, None]
    freq = base ** (-2.0 * np.arange(d // 2, dtype=np.float64) / d)[None, :]
    ang = pos * freq
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct query rows: always 0, 127, 128, N-1 (when they exist),
    the rest uniform without replacement."""
    must = [r for r in (0, 127, 128, N - 1) if 0 <= r < N]
    rng = np.random.Generator(np.random.PCG64([seed, 300]))
    count = min(count, N)
    pool = np.setdiff1d(np.arange(N), np.array(must, dtype=np.int64))
    extra = rng.choice(pool, size=max(0, count - len(set(must))), replace=False) if pool.size else []
    return np.unique(np.concatenate([np.array(must, dtype=np.int64), np.asarray(extra, dtype=np.int64)]))


def sweep_configs():
    """(name, B, H, N, d, seed) for the 16K-token sweep."""
    out = []
    idx = 0
    for (H, d) in SWEEP_HD:
        for N in SWEEP_N:
            out.append((f"sweep_N{N}_d{d}", TOTAL_TOKENS // N, H, N, d, 2 + idx))
            idx += 1
    return out


TINY = dict(name="tiny", B=1, H=2, N=128, d=64, seed=0, scale=1.0 / 8.0)
MID = dict(name="mid", B=4, H=16, N=2048, d=128, seed=1, scale=1.0 / math.sqrt(128))
LONG = dict(name="long", B=1, H=16, N=65536, d=128, seed=5, scale=1.0 / math.sqrt(128))


def flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Forward FLOP count 4*B*H*N^2*d, halved for causal (the pages' convention)."""
    f = 4.0 * B * H * N * N * d
    return f / 2.0 if causal else f
