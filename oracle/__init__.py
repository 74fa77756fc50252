"""FP64 CPU oracle for C = alpha*A*B + beta*C0 (row-major FP32 operands).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``, never by
the product package.  It shares no code with the CUDA library; the only module
both sides use is the seeded input generator, which holds none of the GEMM
arithmetic.

Contents
--------
* ``sgemm_f64`` / ``sgemm_f64_sampled`` -- the definition C_ij = sum_t A_it
  B_tj (hatrix.site "GEMM优化原理", section 问题定义) accumulated in FP64 in
  increasing t, plus BLAS alpha/beta, in plain C (``sgemm_oracle.c``).
* ``within_tolerance`` -- the FP32 acceptance bound
  ``|C - r| <= 1e-5 * sum_t |A_it||B_tj| + 1e-6 * |beta C0_ij|``.  Summation
  order changes the last bits of a float result (aerisun.top "GPU 访存与计算
  优化", the note closing section "Reduce 的分层归约"), so real-valued results
  are compared within a bound rather than bit for bit.
* ``tiling_counts`` -- the tile bookkeeping of hatrix.site "GEMM优化原理"
  (sections 问题定义, 基于 shared memory 计算, 基于 register 计算 and
  一个具体的例子): grid sizes, threads, iterations and the read counts of the
  three storage levels.
* ``sum_f64`` / ``sum_within_tolerance`` -- the array sum s = sum_i x_i of
  aerisun.top "GPU 访存与计算优化" (section "Reduce 的分层归约"), in FP64, and
  the bound gamma_h * sum_i |x_i| every FP32 summation tree of depth h meets
  (h additions on the longest chain, each rounding by at most u = 2^-24).
* ``ideal_intensity`` / ``cta_intensity`` -- the arithmetic-intensity formulas
  of aerisun.top "GPU 访存与计算优化" (sections "GEMM 的理想复用与实际访存" and
  "Shared Tiling 与 block 内复用").

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, exact integer brute force, a library cross-check and the numbers the
pages print (``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None


def lib_path() -> str:
    return os.path.join(_BUILD, f"liboracle_{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compiles the C oracle with gcc (OpenMP, no FP contraction)."""
    out = lib_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            i64, f64, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.oracle_sgemm_f64.argtypes = [i64, i64, i64, f64, vp, i64, vp, i64, f64, vp, i64,
                                             vp, vp, vp, i64, i64, ci]
            lib.oracle_sgemm_f64.restype = None
            lib.oracle_sgemm_f64_sampled.argtypes = [i64, f64, vp, i64, vp, i64, f64, vp, i64,
                                                     i64, vp, vp, vp, vp, ci]
            lib.oracle_sgemm_f64_sampled.restype = None
            lib.oracle_sum_f64.argtypes = [vp, i64, vp, vp]
            lib.oracle_sum_f64.restype = None
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ci
            _LIB = lib
        return _LIB


def max_threads() -> int:
    return int(_lib().oracle_max_threads())


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _as_f32(a, rows, ld):
    a = np.ascontiguousarray(a, dtype=np.float32)
    if rows > 0 and a.size < (rows - 1) * ld + 1:
        raise ValueError("operand smaller than its (rows, ld) extent")
    return a


def sgemm_f64(m, n, k, alpha, A, lda, B, ldb, beta, C0, ldc, *,
              rows: Optional[tuple] = None, nthreads: int = 0):
    """Returns (R, E, Rf): the FP64 result r_ij, the error scale
    E_ij = sum_t |A_it||B_tj| and r rounded to FP32, each (rows) x n.

    ``rows=(r0, r1)`` evaluates only output rows r0..r1-1."""
    r0, r1 = (0, m) if rows is None else rows
    A = _as_f32(A, m, lda)
    B = _as_f32(B, k, ldb)
    C0 = _as_f32(C0, m, ldc) if beta != 0.0 else None
    R = np.empty((r1 - r0, n), dtype=np.float64)
    E = np.empty((r1 - r0, n), dtype=np.float64)
    Rf = np.empty((r1 - r0, n), dtype=np.float32)
    if r1 > r0 and n > 0:
        _lib().oracle_sgemm_f64(m, n, k, float(alpha), _ptr(A), lda, _ptr(B), ldb, float(beta),
                                _ptr(C0), ldc, _ptr(R), _ptr(E), _ptr(Rf), r0, r1, nthreads)
    return R, E, Rf


def sgemm_f64_sampled(k, alpha, A, lda, B, ldb, beta, C0, ldc, rows, cols, *,
                      nthreads: int = 0):
    """(R, E) at the coordinates (rows[s], cols[s]) only."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    C0 = np.ascontiguousarray(C0, dtype=np.float32) if beta != 0.0 else None
    R = np.empty(rows.shape[0], dtype=np.float64)
    E = np.empty(rows.shape[0], dtype=np.float64)
    if rows.shape[0]:
        _lib().oracle_sgemm_f64_sampled(k, float(alpha), _ptr(A), lda, _ptr(B), ldb, float(beta),
                                        _ptr(C0), ldc, rows.shape[0], _ptr(rows), _ptr(cols),
                                        _ptr(R), _ptr(E), nthreads)
    return R, E


def problem_f64(p, **kw):
    """``sgemm_f64`` on a ``dense_fp32_gemm_06_gb300.inputs.Problem``."""
    return sgemm_f64(p.m, p.n, p.k, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta, p.C0, p.ldc, **kw)


def problem_f64_sampled(p, rows, cols, **kw):
    return sgemm_f64_sampled(p.k, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta, p.C0, p.ldc,
                             rows, cols, **kw)


# Acceptance bound for real-valued FP32 results.
TOL_REL_E = 1e-5
TOL_REL_BETA_C0 = 1e-6


def tolerance(E, beta, C0_vals):
    """Allowed |C - r| per element: 1e-5 * E + 1e-6 * |beta * C0|."""
    bound = TOL_REL_E * np.asarray(E, dtype=np.float64)
    if beta != 0.0:
        bound = bound + TOL_REL_BETA_C0 * np.abs(beta * np.asarray(C0_vals, dtype=np.float64))
    return bound


def within_tolerance(C, R, E, beta, C0_vals):
    """(ok, worst_ratio, index): ok when every |C - R| <= tolerance and C is
    finite; worst_ratio is max |C - R| / tolerance (inf where the bound is 0
    and the values differ)."""
    C = np.asarray(C, dtype=np.float64)
    R = np.asarray(R, dtype=np.float64)
    if C.size == 0:
        return True, 0.0, None
    diff = np.abs(C - R)
    bound = tolerance(E, beta, C0_vals)
    finite = np.isfinite(C)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(diff == 0.0, 0.0, diff / bound)
    ratio = np.where(finite, ratio, np.inf)
    idx = int(np.argmax(ratio))
    worst = float(ratio.flat[idx])
    return bool(np.all(finite) and np.all(diff <= bound)), worst, np.unravel_index(idx, C.shape)


def tiling_counts(m, n, k, bm, bn, bk, rm, rn):
    """Tile bookkeeping of the two-level blocking (aligned case: every size
    divides evenly, as the page restricts itself to).

    M = m/bm, N = n/bn, K = k/bk thread-block grid and big iterations,
    X = bm/rm, Y = bn/rn threads per block; bk small iterations of rm*rn FFMA
    each; per big iteration a block moves bm*bk + bk*bn elements from global
    to shared memory.  Read counts over the whole product:
    global mnk(1/bm + 1/bn), shared mnk(1/rm + 1/rn), register 2mnk
    (naive: 2mnk global reads)."""
    for v, d in ((m, bm), (n, bn), (k, bk), (bm, rm), (bn, rn)):
        if d <= 0 or v % d:
            raise ValueError("tiling_counts covers the evenly dividing case only")
    M, N, K = m // bm, n // bn, k // bk
    X, Y = bm // rm, bn // rn
    return dict(
        M=M, N=N, K=K, X=X, Y=Y,
        blocks=M * N,
        c_elements_per_block=bm * bn,
        threads_per_block=X * Y,
        outputs_per_thread=rm * rn,
        big_iterations=K,
        small_iterations=bk,
        ffma_per_small_iteration=rm * rn,
        a_elements_per_big_iteration=bm * bk,
        b_elements_per_big_iteration=bk * bn,
        naive_global_reads=2 * m * n * k,
        global_reads=M * N * K * (bm * bk + bk * bn),
        shared_reads=M * N * K * X * Y * bk * (rm + rn),
        register_reads=M * N * K * X * Y * 2 * rm * rn * bk,
    )


def ideal_intensity(m, n, k, bytes_per_elem=4, c_read=False):
    """FLOP per DRAM byte when every operand is read once and C written once
    (2mnk / (4(mk + kn + mn))); ``c_read=True`` also counts reading C0."""
    mn = m * n * (2 if c_read else 1)
    return 2.0 * m * n * k / (bytes_per_elem * (m * k + k * n + mn))


def cta_intensity(BM, BN, bytes_per_elem=4):
    """FLOP per byte a BM x BN output tile does on one BK-deep slab it loads
    once: 2*BM*BN*BK / (4*(BM*BK + BK*BN)) = BM*BN / (2*(BM + BN)) for FP32."""
    return 2.0 * BM * BN / (bytes_per_elem * (BM + BN))


def sum_f64(x):
    """(s, a): the FP64 sum of the float32 values x and the sum of |x|."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    s = ctypes.c_double(0.0)
    a = ctypes.c_double(0.0)
    _lib().oracle_sum_f64(_ptr(x) if x.size else None, x.size, ctypes.byref(s), ctypes.byref(a))
    return s.value, a.value


def sum_tolerance(abs_sum, depth):
    """gamma_h * sum|x| with gamma_h = h u / (1 - h u), u = 2^-24: the error
    bound of any FP32 summation whose longest chain has h additions."""
    u = 2.0 ** -24
    hu = depth * u
    return hu / (1.0 - hu) * abs_sum


def sum_within_tolerance(got, s, abs_sum, depth):
    return bool(np.isfinite(got)) and abs(float(got) - s) <= sum_tolerance(abs_sum, depth)
