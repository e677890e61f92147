"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the stencil ops: it only draws numbers.
Every tensor is a flat fp32 array filled chunk by chunk; chunk ``j`` of the
tensor with stream id ``stream`` under seed ``seed`` is drawn from
``numpy.random.default_rng([seed, stream, j])`` (PCG64 seeded through
SeedSequence).  The value at any flat index therefore depends only on
(seed, stream, index), never on the thread count, so a caller can regenerate
one plane of a huge tensor without drawing the rest, and chunks can be drawn
in parallel (NumPy releases the GIL while filling).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 20  # elements per independently seeded chunk


def _draw(dist: tuple, rng: np.random.Generator, n: int) -> np.ndarray:
    kind = dist[0]
    if kind == "uniform":
        lo, hi = float(dist[1]), float(dist[2])
        u = rng.random(n, dtype=np.float32)
        return (np.float32(lo) + np.float32(hi - lo) * u).astype(np.float32, copy=False)
    if kind == "normal":
        std = float(dist[1]) if len(dist) > 1 else 1.0
        v = rng.standard_normal(n, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        return v
    if kind == "const":
        return np.full(n, np.float32(dist[1]), dtype=np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def generate_range(dist: tuple, seed: int, stream: int, start: int, stop: int) -> np.ndarray:
    """Flat elements [start, stop) of the tensor (seed, stream, dist)."""
    out = np.empty(max(stop - start, 0), dtype=np.float32)
    pos = start
    while pos < stop:
        j = pos // CHUNK
        c0 = j * CHUNK
        end = min(stop, c0 + CHUNK)
        block = _draw(dist, np.random.default_rng([seed, stream, j]), end - c0)
        out[pos - start:end - start] = block[pos - c0:]
        pos = end
    return out


def generate(dist: tuple, shape, seed: int, stream: int, out: np.ndarray | None = None,
             threads: int | None = None) -> np.ndarray:
    """Whole tensor of ``shape`` (C order, fp32).  ``out`` may be a preallocated
    (e.g. pinned) fp32 array viewed through NumPy."""
    n = int(math.prod(shape))
    if out is None:
        out = np.empty(n, dtype=np.float32)
    flat = out.reshape(-1)
    if flat.size != n or flat.dtype != np.float32:
        raise ValueError("output buffer has the wrong size or dtype")
    nchunks = (n + CHUNK - 1) // CHUNK

    def fill(j):
        c0 = j * CHUNK
        c1 = min(c0 + CHUNK, n)
        flat[c0:c1] = _draw(dist, np.random.default_rng([seed, stream, j]), c1 - c0)

    if threads is None:
        threads = min(os.cpu_count() or 1, 32)
    if nchunks <= 1 or threads <= 1:
        for j in range(nchunks):
            fill(j)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)
