"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds none of the method's arithmetic: it draws standard-normal
Q, K, V, rounds them to bf16 and returns the bf16 bit patterns, so that the
CPU oracle and the GPU path read the very same bytes.

Recipe (one seed):
  rng = numpy.random.default_rng(seed)
  Q, K, V = rng.standard_normal([B, H, S, D], float32) drawn in that order,
  rounded to bf16 (round-to-nearest-even) and kept as uint16 bit patterns.
Rollback-stress variant: after Q, K, V, draw ``rng.random([B, H, S])`` and
multiply every K row at key position j >= stress_from whose draw is < frac by
8 (exact in bf16), so that later tiles pass the frozen reference.
"""
from __future__ import annotations

import numpy as np
import torch


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def qkv(B: int, H: int, S: int, D: int, seed: int = 0, stress_from: int | None = None,
        stress_frac: float = 0.01, stress_mult: float = 8.0, chunk: int = 1 << 26):
    """Return (q, k, v) bf16 bit patterns, each uint16 [B, H, S, D]."""
    rng = np.random.default_rng(seed)
    out = []
    n = B * H * S * D
    for _ in range(3):
        bits = np.empty(n, np.uint16)
        # draw in chunks so that huge shapes do not need a float32 copy of all
        for i in range(0, n, chunk):
            m = min(chunk, n - i)
            bits[i:i + m] = to_bf16_bits(rng.standard_normal(m, dtype=np.float32))
        out.append(bits.reshape(B, H, S, D))
    q, k, v = out
    if stress_from is not None:
        mask = rng.random((B, H, S)) < stress_frac
        mask[:, :, :stress_from] = False
        kf = bf16_bits_to_f32(k[mask]) * np.float32(stress_mult)
        k[mask] = to_bf16_bits(kf)
    return q, k, v


def sample_rows(B: int, H: int, S: int, n_random: int = 1024, seed: int = 0) -> np.ndarray:
    """Row subsample for parity at full size: n_random random rows drawn with
    seed+1000, plus every row of the first and last 128-row query tile of the
    first and the last head.  Returns sorted unique global row indices."""
    rng = np.random.default_rng(seed + 1000)
    BH = B * H
    rnd = rng.integers(0, BH * S, size=n_random)
    last0 = ((S - 1) // 128) * 128
    fixed = []
    for bh in (0, BH - 1):
        fixed.append(bh * S + np.arange(0, min(128, S)))
        fixed.append(bh * S + np.arange(last0, S))
    return np.unique(np.concatenate([rnd] + fixed)).astype(np.int64)
