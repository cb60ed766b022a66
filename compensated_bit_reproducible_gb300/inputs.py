"""Seeded synthetic inputs shared by the tests and the benchmark.

This module only draws numbers: it holds none of the summation or variance
arithmetic, so the CUDA path and the CPU oracle can both consume its arrays.
Every generator is `numpy.random.default_rng(seed)` based and returns host
numpy arrays; shapes, value distributions and structure follow the workloads
the pages measure (the SyclReproSum's 100M-element sums, the variance
note's D1-D4 datasets, identical-value rows and [4096, 4096] speed array).
"""
from __future__ import annotations

import numpy as np


def quickstart_f64() -> np.ndarray:
    """5 pairs (1e16, -1e16) then 10000 ones (SyclReproSum, Quick Start)."""
    return np.array([1e16, -1e16] * 5 + [1.0] * 10000, dtype=np.float64)


def permuted(x: np.ndarray, seed: int) -> np.ndarray:
    return x[np.random.default_rng(seed).permutation(x.size)]


def thousandth_f32(n: int = 1_000_000) -> np.ndarray:
    """n copies of 0.001f (Kahan's Summation Formula)."""
    return np.full(n, np.float32(0.001), dtype=np.float32)


def normal_f32(n: int, seed: int = 1, spikes: bool = False) -> np.ndarray:
    """N(0, 1) float32; with `spikes`, 1% of entries (without replacement)
    scaled by 1e6 with a random sign."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n, dtype=np.float32)
    if spikes and n:
        k = max(1, n // 100)
        idx = rng.choice(n, size=k, replace=False)
        sign = np.where(rng.random(k) < 0.5, -1.0, 1.0).astype(np.float32)
        x[idx] = (x[idx] * np.float32(1e6) * sign).astype(np.float32)
    return x


def wide_f64(n: int, seed: int = 2, cancel_frac: float = 0.10) -> np.ndarray:
    """s * 2^u with s = +-1 and u ~ U(-60, 60); `cancel_frac` of the entries
    form exactly cancelling (v, -v) pairs at random positions."""
    rng = np.random.default_rng(seed)
    u = rng.uniform(-60.0, 60.0, n)
    s = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    x = s * np.exp2(u)
    m = int(n * cancel_frac) // 2
    if m:
        idx = rng.choice(n, size=2 * m, replace=False)
        v = x[idx[:m]]
        x[idx[m:]] = -v
    return x


def inject_specials(x: np.ndarray, kind: str, seed: int = 7) -> np.ndarray:
    """Copy of x with special values at random positions: 'nan' (NaNs with
    random payloads and signs), 'pinf', 'pninf' (+Inf and -Inf)."""
    y = x.copy()
    rng = np.random.default_rng(seed)
    n = y.size
    pos = rng.choice(n, size=min(n, 4), replace=False)
    if kind == "nan":
        if y.dtype == np.float64:
            bits = y.view(np.uint64)
            for p in pos[:3]:
                payload = int(rng.integers(1, 1 << 51))
                sign = int(rng.integers(0, 2)) << 63
                bits[p] = np.uint64(sign | (0x7FF << 52) | payload)
        else:
            bits = y.view(np.uint32)
            for p in pos[:3]:
                payload = int(rng.integers(1, 1 << 22))
                sign = int(rng.integers(0, 2)) << 31
                bits[p] = np.uint32(sign | (0xFF << 23) | payload)
    elif kind == "pinf":
        y[pos[0]] = np.inf
    elif kind == "pninf":
        y[pos[0]] = np.inf
        y[pos[1]] = -np.inf
    else:
        raise ValueError(kind)
    return y


def var_datasets(seed: int = 0):
    """The variance note's four dataset shapes (section 3), float32:
    (name, array, axis)."""
    rng = np.random.default_rng(seed)
    d1 = rng.normal(1000.0, 0.01, (1000, 64)).astype(np.float32)
    d2 = rng.normal(10000.0, 1.0, (64, 1000)).astype(np.float32)
    d3 = rng.normal(0.0, 1.0, (1000, 64)).astype(np.float32)
    d4 = rng.normal(1e6, 1.0, (1000, 64)).astype(np.float32)
    return [("D1", d1, 0), ("D2", d2, 1), ("D3", d3, 0), ("D4", d4, 0)]


def identical_rows(cols: int = 4096) -> np.ndarray:
    """[8, cols] float32, row r filled with (1, 1e10, 1e30, 1e38)[r % 4]."""
    vals = np.array([1.0, 1e10, 1e30, 1e38], dtype=np.float32)
    return np.repeat(vals[np.arange(8) % 4][:, None], cols, axis=1).astype(np.float32)


def offset_rows(rows: int = 4096, cols: int = 4096, seed: int = 3, heavy: bool = False) -> np.ndarray:
    """Row offset U[1e3, 1e5] plus N(0, 1) noise; with `heavy`, the
    gradient-like variant 1e-3 * Student-t(df=3) without offset."""
    rng = np.random.default_rng(seed)
    if heavy:
        return (1e-3 * rng.standard_t(3, (rows, cols))).astype(np.float32)
    off = rng.uniform(1e3, 1e5, (rows, 1))
    return (off + rng.standard_normal((rows, cols))).astype(np.float32)
