"""The projection check the full-size GPU parity tests use
(`gpu_util.projection_ratios`, Freivalds' check against the per-element FP32
bound), pinned on the CPU: a C within the bound everywhere passes, and a C
with one tile gone wrong -- zeroed, taken from its neighbour, a k part or
beta C0 added twice, rows swapped inside it -- fails, on both its rows and its
columns."""
import numpy as np
import pytest
import torch

from dense_fp32_gemm_06_gb300 import inputs
from gpu_util import projection_ratios

M, N, K = 512, 768, 384
TM, TN = 128, 256          # one tensor-core tile of C


@pytest.fixture(scope="module")
def problem():
    p = inputs.make_problem(M, N, K, alpha=1.25, beta=0.5, seed=11, a="normal", b="uniform", c="uniform")
    A = torch.from_numpy(np.ascontiguousarray(p.A[:, :K]))
    B = torch.from_numpy(np.ascontiguousarray(p.B[:, :N]))
    C0 = torch.from_numpy(np.ascontiguousarray(p.C0[:, :N]))
    exact = p.alpha * (A.double() @ B.double()) + p.beta * C0.double()
    return p, A, B, C0, exact


def ratios(problem, C):
    p, A, B, C0, _ = problem
    return projection_ratios(A, B, C0, C, p.alpha, p.beta, seed=5)


def test_exact_product_passes(problem):
    C = problem[4].float()      # the exact result rounded once to FP32
    rx, ry = ratios(problem, C)
    assert rx <= 1.0 and ry <= 1.0


def test_fp32_accumulation_passes(problem):
    """A plain FP32 product (well inside the bound) passes too."""
    p, A, B, C0, _ = problem
    C = p.alpha * (A @ B) + p.beta * C0
    rx, ry = ratios(problem, C)
    assert rx <= 1.0 and ry <= 1.0


def _tile(C, ti, tj):
    return C[ti * TM:(ti + 1) * TM, tj * TN:(tj + 1) * TN]


def _zeroed(problem, C):
    _tile(C, 1, 1).zero_()


def _neighbour(problem, C):
    _tile(C, 2, 1).copy_(_tile(C, 2, 2))


def _k_part_twice(problem, C):
    p, A, B, _, _ = problem
    rows, cols = slice(3 * TM, 4 * TM), slice(0, TN)
    C[rows, cols] += p.alpha * (A[rows, : K // 2].double() @ B[: K // 2, cols].double()).float()


def _beta_twice(problem, C):
    p, _, _, C0, _ = problem
    _tile(C, 0, 2).add_(p.beta * _tile(C0, 0, 2))


def _rows_swapped(problem, C):
    t = _tile(C, 1, 0)
    t.copy_(t.flip(0))


@pytest.mark.parametrize("mutate", [_zeroed, _neighbour, _k_part_twice, _beta_twice, _rows_swapped],
                         ids=["zeroed", "neighbour", "k_part_twice", "beta_twice", "rows_swapped"])
def test_one_wrong_tile_fails(problem, mutate):
    C = problem[4].float().clone()
    mutate(problem, C)
    rx, ry = ratios(problem, C)
    assert rx > 1.0 and ry > 1.0, (rx, ry)
