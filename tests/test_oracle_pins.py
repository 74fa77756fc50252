"""Pins the FP64 oracle to facts other than itself (CPU only).

Each pin is a function of an oracle callable
``f(m, n, k, alpha, A, lda, B, ldb, beta, C0, ldc) -> (R, E)`` so that the
same pins can be run on planted mutants (a transposed operand, a dropped
beta term, a wrong sign, an off-by-one in t, a wrong leading dimension, ...)
and shown to reject every one of them.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_06_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def real_oracle(m, n, k, alpha, A, lda, B, ldb, beta, C0, ldc):
    R, E, _ = oracle.sgemm_f64(m, n, k, alpha, A, lda, B, ldb, beta, C0, ldc)
    return R, E


def rng_int(shape, seed, lo=-4, hi=4):
    return np.random.default_rng(seed).integers(lo, hi + 1, size=shape).astype(np.float32)


# --------------------------------------------------------------------------- pins

def pin_identity(f):
    """A = I (m = k): r = alpha*B + beta*C0 exactly, E = |B|."""
    k, n = 37, 53
    B = inputs.draw_matrix("uniform", 11, 0, k, n)
    C0 = inputs.draw_matrix("normal", 11, 10_000, k, n)
    A = np.eye(k, dtype=np.float32)
    for alpha, beta in ((1.0, 0.0), (1.5, 0.5), (-2.0, 1.0)):
        R, E = f(k, n, k, alpha, A, k, B, n, beta, C0, n)
        want = alpha * B.astype(np.float64) + (beta * C0.astype(np.float64) if beta else 0.0)
        if not np.array_equal(R, want) or not np.array_equal(E, np.abs(B.astype(np.float64))):
            return False
    return True


def pin_permutation(f):
    """A a permutation: rows of B permuted; B a permutation: columns of A permuted."""
    m = k = n = 41
    perm = np.random.default_rng(5).permutation(k)
    P = np.zeros((k, k), dtype=np.float32)
    P[np.arange(k), perm] = 1.0
    X = inputs.draw_matrix("uniform", 12, 0, k, k)
    C0 = np.zeros((m, n), dtype=np.float32)
    R1, _ = f(m, n, k, 1.0, P, k, X, n, 0.0, C0, n)
    R2, _ = f(m, n, k, 1.0, X, k, P, n, 0.0, C0, n)
    inv = np.argsort(perm)
    return (np.array_equal(R1, X[perm, :].astype(np.float64))
            and np.array_equal(R2, X[:, inv].astype(np.float64)))


def pin_rank1(f):
    """A = u 1^T, B = 1 v^T: C_ij = k u_i v_j (integers: exact)."""
    m, n, k = 19, 23, 29
    u = rng_int((m,), 1, -9, 9)
    v = rng_int((n,), 2, -9, 9)
    A = np.repeat(u[:, None], k, axis=1).astype(np.float32)
    B = np.repeat(v[None, :], k, axis=0).astype(np.float32)
    R, E = f(m, n, k, 1.0, A, k, B, n, 0.0, np.zeros((m, n), np.float32), n)
    want = k * np.outer(u.astype(np.float64), v.astype(np.float64))
    return np.array_equal(R, want) and np.array_equal(E, np.abs(want))


def pin_linearity(f):
    """r(alpha, beta) = alpha * r(1, 0) + beta * C0, exact on integer twins."""
    m, n, k = 31, 17, 45
    A, B, C0 = rng_int((m, k), 3), rng_int((k, n), 4), rng_int((m, n), 5)
    R10, _ = f(m, n, k, 1.0, A, k, B, n, 0.0, C0, n)
    for alpha, beta in itertools.product((1.5, 2.0), (0.5, 1.0)):
        R, _ = f(m, n, k, alpha, A, k, B, n, beta, C0, n)
        if not np.array_equal(R, alpha * R10 + beta * C0.astype(np.float64)):
            return False
    return True


def pin_bruteforce(f, sizes=range(1, 9)):
    """Every m, n, k in 1..8 on integers in {-4..4} against a pure-Python
    integer triple loop: exact equality (and E = sum |a||b| exactly)."""
    seed = 100
    for m, n, k in itertools.product(sizes, sizes, sizes):
        seed += 1
        A, B, C0 = rng_int((m, k), seed), rng_int((k, n), seed + 7), rng_int((m, n), seed + 13)
        Ai, Bi, Ci = A.astype(int).tolist(), B.astype(int).tolist(), C0.astype(int).tolist()
        R, E = f(m, n, k, 2.0, A, k, B, n, -1.0, C0, n)
        for i in range(m):
            for j in range(n):
                acc = 0
                err = 0
                for t in range(k):
                    acc += Ai[i][t] * Bi[t][j]
                    err += abs(Ai[i][t]) * abs(Bi[t][j])
                if R[i, j] != 2 * acc - Ci[i][j] or E[i, j] != err:
                    return False
    return True


def pin_library(f):
    """torch.matmul in FP64 (CPU) on real-valued inputs, up to 512:
    |r - torch| <= 1e-12 * E (both are FP64 sums of the same products)."""
    for (m, n, k), seed in (((512, 384, 512), 21), ((100, 7, 333), 22), ((1, 512, 1), 23)):
        A = inputs.draw_matrix("normal", seed, 0, m, k)
        B = inputs.draw_matrix("uniform", seed, 2 * m * k, k, n)
        C0 = inputs.draw_matrix("uniform", seed, 4 * m * k + 4 * k * n, m, n)
        R, E = f(m, n, k, 0.75, A, k, B, n, -0.25, C0, n)
        T = (0.75 * (torch.from_numpy(A).double() @ torch.from_numpy(B).double())
             - 0.25 * torch.from_numpy(C0).double()).numpy()
        Eref = (torch.from_numpy(np.abs(A)).double() @ torch.from_numpy(np.abs(B)).double()).numpy()
        if not np.all(np.abs(R - T) <= 1e-12 * (0.75 * Eref + 0.25 * np.abs(C0))):
            return False
        if not np.allclose(E, Eref, rtol=1e-13, atol=0.0):
            return False
    return True


def pin_leading_dims(f):
    """Padded leading dimensions (padding = NaN) give the compact result."""
    m, n, k = 13, 9, 11
    A = inputs.draw_matrix("int", 7, 0, m, k, ld=k + 5)
    B = inputs.draw_matrix("int", 7, 1000, k, n, ld=n + 3)
    C0 = inputs.draw_matrix("int", 7, 2000, m, n, ld=n + 7)
    R, E = f(m, n, k, 1.5, A, k + 5, B, n + 3, 0.5, C0, n + 7)
    Rc, Ec = f(m, n, k, 1.5, np.ascontiguousarray(A[:, :k]), k, np.ascontiguousarray(B[:, :n]), n,
               0.5, np.ascontiguousarray(C0[:, :n]), n)
    return np.array_equal(R, Rc) and np.array_equal(E, Ec) and np.all(np.isfinite(R))


def pin_quick_returns(f):
    """beta = 0 never reads C0 (NaN C0 gives a finite result); alpha = 0 and
    k = 0 give beta * C0 without reading A or B (NaN A, B)."""
    m, n, k = 6, 5, 4
    A, B = rng_int((m, k), 31), rng_int((k, n), 32)
    C0 = rng_int((m, n), 33)
    Rn, _ = f(m, n, k, 1.0, A, k, B, n, 0.0, np.full((m, n), np.nan, np.float32), n)
    nanA, nanB = np.full((m, k), np.nan, np.float32), np.full((k, n), np.nan, np.float32)
    Ra, Ea = f(m, n, k, 0.0, nanA, k, nanB, n, 2.0, C0, n)
    Rk, Ek = f(m, n, 0, 1.0, nanA, 1, nanB, n, 2.0, C0, n)
    want = 2.0 * C0.astype(np.float64)
    return (np.all(np.isfinite(Rn)) and np.array_equal(Ra, want) and np.array_equal(Rk, want)
            and not np.any(Ea) and not np.any(Ek))


PINS = [pin_identity, pin_permutation, pin_rank1, pin_linearity, pin_bruteforce,
        pin_library, pin_leading_dims, pin_quick_returns]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(pin):
    assert pin(real_oracle)


# ------------------------------------------------------------------ planted mistakes
# Each mutant is a plausible slip in writing the definition; the pins above
# must reject every one of them.

def _ref_loops(m, n, k, alpha, A, lda, B, ldb, beta, C0, ldc, *, transA=False, swap=False,
               drop_beta=False, beta_sign=1.0, t_stop=0, use_lda=None, abs_e=True,
               ignore_alpha=False, read_c0_always=False, skip_alpha_zero=True):
    A2 = np.asarray(A, np.float64).reshape(-1)
    B2 = np.asarray(B, np.float64).reshape(-1)
    C2 = np.asarray(C0, np.float64).reshape(-1)
    lda_ = use_lda(lda, k) if use_lda else lda
    R = np.zeros((m, n))
    E = np.zeros((m, n))
    use_ab = not (skip_alpha_zero and (alpha == 0.0 or k == 0))
    for i in range(m):
        for j in range(n):
            acc = err = 0.0
            if use_ab:
                for t in range(k - t_stop):
                    if swap:
                        a, b = B2[i * ldb + t] if i * ldb + t < B2.size else 0.0, A2[t * lda_ + j] if t * lda_ + j < A2.size else 0.0
                    elif transA:
                        a, b = A2[t * lda_ + i], B2[t * ldb + j]
                    else:
                        a, b = A2[i * lda_ + t], B2[t * ldb + j]
                    acc += a * b
                    err += abs(a) * abs(b) if abs_e else a * b
            v = (acc if ignore_alpha else alpha * acc) if use_ab else 0.0
            if (beta != 0.0 or read_c0_always) and not drop_beta:
                v += beta_sign * beta * C2[i * ldc + j]
            R[i, j] = v
            E[i, j] = err
    return R, E


MUTANTS = {
    "transposed_A": dict(transA=True),
    "operands_swapped": dict(swap=True),
    "dropped_beta": dict(drop_beta=True),
    "beta_sign": dict(beta_sign=-1.0),
    "last_t_dropped": dict(t_stop=1),
    "lda_assumed_k": dict(use_lda=lambda lda, k: k),
    "error_scale_without_abs": dict(abs_e=False),
    "alpha_ignored": dict(ignore_alpha=True),
    "c0_read_when_beta_zero": dict(read_c0_always=True),
    "alpha_zero_reads_A": dict(skip_alpha_zero=False),
}


def _guarded(pin, f):
    try:
        with np.errstate(all="ignore"):
            return pin(f)
    except (IndexError, ValueError):
        return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name):
    kw = MUTANTS[name]

    def mutant(*args):
        return _ref_loops(*args, **kw)

    # brute force over 1..4 keeps the pure-Python mutant fast; the library
    # pin is skipped (512^3 in Python loops) -- every mutant must already
    # fail one of the others.
    pins = [p for p in PINS if p not in (pin_bruteforce, pin_library)]
    pins.append(lambda f: pin_bruteforce(f, sizes=range(1, 5)))
    assert not all(_guarded(p, mutant) for p in pins), f"no pin rejects mutant {name}"


def test_reference_loops_without_mistake_pass():
    """The unmutated Python loops pass the same pins, so the mutant test is
    rejecting the planted mistakes, not the loop harness."""
    pins = [p for p in PINS if p not in (pin_bruteforce, pin_library)]
    assert all(p(lambda *a: _ref_loops(*a)) for p in pins)


# ------------------------------------------------------------------ sampled oracle

def test_sampled_matches_full():
    p = inputs.workload("1000x1500x777")
    rows, cols = inputs.sample_indices(p.m, p.n, 500, seed=1002)
    R, E, _ = oracle.problem_f64(p, rows=(0, p.m))
    Rs, Es = oracle.problem_f64_sampled(p, rows, cols)
    assert np.array_equal(Rs, R[rows, cols]) and np.array_equal(Es, E[rows, cols])


def test_row_slab_matches_full():
    p = inputs.workload("256^3")
    R, E, Rf = oracle.problem_f64(p)
    R2, E2, Rf2 = oracle.problem_f64(p, rows=(64, 130))
    assert np.array_equal(R2, R[64:130]) and np.array_equal(Rf2, Rf[64:130])
    assert np.array_equal(Rf, R.astype(np.float32))


def test_tolerance_function():
    E = np.array([1.0, 2.0, 0.0])
    R = np.array([0.0, 0.0, 1.0])
    ok, worst, _ = oracle.within_tolerance(R + np.array([1e-5, 1.9e-5, 0.0]), R, E, 0.0, None)
    assert ok and worst <= 1.0
    ok, _, _ = oracle.within_tolerance(R + np.array([1.1e-5, 0.0, 0.0]), R, E, 0.0, None)
    assert not ok
    # beta term: 1e-6 * |beta C0|
    ok, _, _ = oracle.within_tolerance(np.array([1.0 + 0.9e-6]), np.array([1.0]), np.array([0.0]),
                                       0.5, np.array([2.0]))
    assert ok
    ok, _, _ = oracle.within_tolerance(np.array([np.nan]), np.array([1.0]), np.array([1.0]), 0.0, None)
    assert not ok


# ------------------------------------------------------------------ pages' printed numbers

def _golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def test_worked_example_tile_arithmetic():
    g = _golden("worked_example_2048.json")
    got = oracle.tiling_counts(**g["inputs"])
    for key, want in g["expected"].items():
        assert got[key] == want, key


def test_read_count_closed_forms():
    m, n, k = 2048, 1024, 512
    for bm, bn, bk, rm, rn in ((128, 128, 8, 8, 8), (64, 128, 16, 4, 8), (256, 64, 32, 16, 4)):
        c = oracle.tiling_counts(m, n, k, bm, bn, bk, rm, rn)
        assert c["global_reads"] * bm * bn == m * n * k * (bm + bn)
        assert c["shared_reads"] * rm * rn == m * n * k * (rm + rn)
        assert c["register_reads"] == 2 * m * n * k == c["naive_global_reads"]


def test_float4_per_thread():
    g = _golden("float4_per_thread.json")
    c = oracle.tiling_counts(**g["inputs"])
    assert c["a_elements_per_big_iteration"] == g["expected"]["a_elements_per_big_iteration"]
    assert c["threads_per_block"] == g["expected"]["threads_per_block"]
    assert c["a_elements_per_big_iteration"] // (4 * c["threads_per_block"]) == \
        g["expected"]["float4_per_thread_per_operand"]


def test_cta_tile_intensity():
    g = _golden("cta_tile_64.json")
    BM, BN, BK = g["inputs"]["BM"], g["inputs"]["BN"], g["inputs"]["BK"]
    assert 4 * (BM * BK + BK * BN) == g["expected"]["smem_bytes"]
    assert BM * BN * BK == g["expected"]["fma"]
    assert 2 * BM * BN * BK == g["expected"]["flop"]
    assert oracle.cta_intensity(BM, BN) == g["expected"]["flop_per_byte"]


def test_ideal_intensity_square_is_n_over_6():
    for n in (6, 600, 2048, 8192):
        assert abs(oracle.ideal_intensity(n, n, n) - n / 6.0) < 1e-9 * n
        assert abs(oracle.ideal_intensity(n, n, n, c_read=True) - n / 8.0) < 1e-9 * n
