"""Seeded synthetic inputs for the SGEMM problem C = alpha*A*B + beta*C.

This module only draws numbers: it holds none of the GEMM arithmetic, so the
CUDA path and the FP64 oracle can both be fed from it without sharing any of
the computation they are compared on.

Generator (counter-based splitmix64)
------------------------------------
Draw ``e`` of the stream for ``seed`` is ``mix(seed + (e + 1) * G)`` with
``G = 0x9E3779B97F4A7C15`` and ``mix`` the splitmix64 finaliser (Steele, Lea
and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014).
That is exactly the sequential splitmix64 stream, indexed so that any slice
of it can be drawn without generating the prefix.

Element ``e`` of a matrix uses draw ``offset + e`` (row-major over the
logical rows x cols, padding excluded).  A problem fills A, then B, then C0,
each starting at an even draw index:

* ``uniform``: ``u = (draw >> 40) * 2^-24`` in [0, 1), value ``2u - 1`` in
  [-1, 1) -- exact in FP32 (24 significant bits).
* ``normal``: Box-Muller in FP64 on the consecutive pair of draws
  ``(2p, 2p+1)`` of the matrix, ``u1 = ((d0 >> 11) + 1) * 2^-53`` in (0, 1],
  ``u2 = (d1 >> 11) * 2^-53``; element ``2p`` gets ``r cos(2 pi u2)`` and
  ``2p+1`` gets ``r sin(2 pi u2)``, ``r = sqrt(-2 ln u1)``, rounded to FP32.
* ``uniform01``: ``u`` itself, in [0, 1) (non-negative operands: every
  partial sum grows, the hardest case for a biased accumulation);
* ``int``: ``floor(9u) - 4`` with ``u`` as for ``uniform`` -- integers in
  {-4..4}, the "integer twin" whose every product and partial sum is exact
  in FP32 while ``16 * k < 2^24``.

The workload shapes (256^3, 2048^3, 1000x1500x777, 8192^3, 16384x128x8192)
are the synthetic dense matrices of the GEMM pages: the 2048^3 size is the
worked example of hatrix.site "GEMM优化原理" (section 一个具体的例子) and the
test size of blog.lightlisten.com "gemm优化" (section 最终结果).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of the splitmix64 stream of ``seed``."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def _u24(draws: np.ndarray) -> np.ndarray:
    return (draws >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)


def _fill(dist: str, seed: int, offset: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    for lo in range(0, count, _CHUNK):
        hi = min(count, lo + _CHUNK)
        if dist == "uniform":
            out[lo:hi] = (_u24(splitmix64(seed, offset + lo, hi - lo)) * 2.0 - 1.0).astype(np.float32)
        elif dist == "uniform01":
            out[lo:hi] = _u24(splitmix64(seed, offset + lo, hi - lo)).astype(np.float32)
        elif dist == "int":
            out[lo:hi] = (np.floor(_u24(splitmix64(seed, offset + lo, hi - lo)) * 9.0) - 4.0).astype(np.float32)
        elif dist == "normal":
            # pairs are aligned to even element indices (lo is a multiple of _CHUNK, which is even)
            plo, phi = lo, hi + (hi - lo) % 2
            d = splitmix64(seed, offset + plo, phi - plo)
            u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
            u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
            r = np.sqrt(-2.0 * np.log(u1))
            z = np.empty(phi - plo, dtype=np.float64)
            z[0::2] = r * np.cos(2.0 * np.pi * u2)
            z[1::2] = r * np.sin(2.0 * np.pi * u2)
            out[lo:hi] = z[: hi - lo].astype(np.float32)
        else:
            raise ValueError(f"unknown distribution {dist!r}")
    return out


def draw_matrix(dist: str, seed: int, offset: int, rows: int, cols: int,
                ld: Optional[int] = None, pad_value: float = float("nan")) -> np.ndarray:
    """A rows x ld FP32 array whose first ``cols`` columns hold draws
    ``offset .. offset + rows*cols - 1`` (row-major); the padding columns
    hold ``pad_value`` (NaN by default, so reading them poisons a result)."""
    ld = cols if ld is None else ld
    if ld < cols:
        raise ValueError("ld < cols")
    vals = _fill(dist, seed, offset, rows * cols).reshape(rows, cols)
    if ld == cols:
        return vals
    out = np.full((rows, ld), pad_value, dtype=np.float32)
    out[:, :cols] = vals
    return out


def _even(x: int) -> int:
    return x + (x & 1)


@dataclasses.dataclass
class Problem:
    """One synthetic SGEMM problem: row-major A (m x lda), B (k x ldb),
    C0 (m x ldc), and the scalars."""
    m: int
    n: int
    k: int
    alpha: float
    beta: float
    A: np.ndarray
    B: np.ndarray
    C0: np.ndarray
    lda: int
    ldb: int
    ldc: int
    seed: int
    dists: tuple


def make_problem(m: int, n: int, k: int, *, alpha: float = 1.0, beta: float = 0.0,
                 seed: int = 0, a: str = "uniform", b: str = "uniform",
                 c: Optional[str] = None, lda: Optional[int] = None,
                 ldb: Optional[int] = None, ldc: Optional[int] = None,
                 pad_value: float = float("nan"),
                 c_fill: float = 0.0) -> Problem:
    """Draws A, then B, then C0 from one splitmix64 stream.

    ``c=None`` leaves C0 at ``c_fill`` (use NaN with beta=0 to check that C0
    is never read)."""
    lda = max(1, k) if lda is None else lda
    ldb = max(1, n) if ldb is None else ldb
    ldc = max(1, n) if ldc is None else ldc
    off_b = _even(m * k)
    off_c = off_b + _even(k * n)
    A = draw_matrix(a, seed, 0, m, k, lda, pad_value)
    B = draw_matrix(b, seed, off_b, k, n, ldb, pad_value)
    if c is None:
        C0 = np.full((m, ldc), c_fill, dtype=np.float32)
        if ldc > n:
            C0[:, n:] = pad_value
    else:
        C0 = draw_matrix(c, seed, off_c, m, n, ldc, pad_value)
    return Problem(m, n, k, float(np.float32(alpha)), float(np.float32(beta)),
                   A, B, C0, lda, ldb, ldc, seed, (a, b, c))


# The five workloads.  ``twin`` swaps every real-valued distribution for the
# integer twin of the same shape (the bit-exact check).
WORKLOADS = {
    "256^3": dict(m=256, n=256, k=256, alpha=1.0, beta=0.0, seed=0, a="uniform", b="uniform", c=None),
    "2048^3": dict(m=2048, n=2048, k=2048, alpha=1.0, beta=0.0, seed=1, a="uniform", b="uniform", c=None),
    "1000x1500x777": dict(m=1000, n=1500, k=777, alpha=1.5, beta=0.5, seed=2, a="uniform", b="uniform", c="normal"),
    "8192^3": dict(m=8192, n=8192, k=8192, alpha=1.0, beta=0.0, seed=3, a="normal", b="normal", c=None),
    "16384x128x8192": dict(m=16384, n=128, k=8192, alpha=1.0, beta=1.0, seed=4, a="uniform", b="uniform", c="uniform"),
}


def workload(name: str, twin: bool = False, **over) -> Problem:
    spec = dict(WORKLOADS[name])
    if twin:
        for key in ("a", "b", "c"):
            if spec[key] is not None:
                spec[key] = "int"
    spec.update(over)
    return make_problem(**spec)


def sample_indices(m: int, n: int, count: int, seed: int, tile_m: int = 128,
                   tile_n: int = 128) -> tuple:
    """``count`` output coordinates drawn from the stream of ``seed``, plus
    the four corners and the last row/column of every partial tile edge.
    Returned as two int64 arrays (rows, cols) without duplicates."""
    d = splitmix64(seed, 0, 2 * count)
    rows = ((d[0::2] >> np.uint64(11)) % np.uint64(m)).astype(np.int64)
    cols = ((d[1::2] >> np.uint64(11)) % np.uint64(n)).astype(np.int64)
    extra_r = [0, 0, m - 1, m - 1]
    extra_c = [0, n - 1, 0, n - 1]
    for r in range(tile_m - 1, m, tile_m):
        extra_r += [r, r]
        extra_c += [0, n - 1]
    for c in range(tile_n - 1, n, tile_n):
        extra_r += [0, m - 1]
        extra_c += [c, c]
    rows = np.concatenate([rows, np.array(extra_r, dtype=np.int64)])
    cols = np.concatenate([cols, np.array(extra_c, dtype=np.int64)])
    key = np.unique(rows * n + cols)
    return key // n, key % n
