"""Column-parallel calls of the CPU oracle for the GPU parity tests.

The oracle computes every token column on its own (column t of Y depends on
column t of X alone, exactly, in fp64), so running it on chunks of the
columns in a thread pool gives the same result as one call over all of them.
ctypes releases the GIL around each C call, so the chunks run on separate
host cores.  This helper only splits the work; the arithmetic stays in the
oracle.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle


def workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def gemm_columns(parent: dict, x_bf16: np.ndarray, chunk: int = 8):
    """(Y, A) of the oracle on every row of x_bf16 ([T, K] bf16 patterns)."""
    x = np.ascontiguousarray(x_bf16)
    T = x.shape[0]
    if T <= chunk or workers() == 1:
        return oracle.gemm_parent(parent, x)
    lib = oracle.load()
    spans = [(i, min(T, i + chunk)) for i in range(0, T, chunk)]
    with ThreadPoolExecutor(max_workers=workers()) as ex:
        parts = list(ex.map(lambda s: oracle.gemm_parent(parent, x[s[0]:s[1]], lib=lib), spans))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def wide_columns(T: int, every: int = 64, extra: int = 16, seed: int = 0) -> np.ndarray:
    """The token columns a wide-T parity test compares: all of them up to
    T = 256; beyond, every `every`-th column (so that each 128-token tile and
    both 64-column halves of its epilogue are covered), the last column and
    `extra` seeded random ones."""
    if T <= 256:
        return np.arange(T)
    rng = np.random.default_rng(seed + T)
    pick = rng.choice(np.arange(1, T - 1), size=extra, replace=False)
    return np.unique(np.concatenate([np.arange(0, T, every), [T - 1], pick]))
