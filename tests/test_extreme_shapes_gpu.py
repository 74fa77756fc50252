"""GPU parity at the extremes of the shape space, on both paths and the
automatic choice, against the FP64 oracle on sampled outputs (plus every
output when there are few): k up to 2^20 (a 1 x 1 x 2^20 dot product and
16 x 16 outputs over 2^20 terms), m or n up to 2^20 with the other two
dimensions tiny, 1-wide problems, and integer twins bit-exact where every
partial sum stays an integer below 2^24."""
import numpy as np
import pytest
import torch

from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import Placed, check_full, check_sampled

pytestmark = pytest.mark.gpu

PATHS = {"ffma": binding.PATH_FFMA, "tf32x3": binding.PATH_TF32X3, "auto": binding.PATH_AUTO}


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _run(p, path, exact=False, samples=4096):
    pl = Placed(p)
    st = pl.run(path)
    assert st == 0, binding.status_string(st)
    C, guard_ok = pl.result()
    assert guard_ok, "a write landed outside the m x n window of C"
    assert pl.inputs_untouched(), "A or B was modified"
    if p.m * p.n <= samples:
        ok, worst, where = check_full(p, C, exact=exact)
    else:
        rows, cols = inputs.sample_indices(p.m, p.n, samples, seed=p.seed + 77)
        # plus the four corners
        rows = np.concatenate([rows, [0, 0, p.m - 1, p.m - 1]])
        cols = np.concatenate([cols, [0, p.n - 1, 0, p.n - 1]])
        ok, worst, where = check_sampled(p, C, rows, cols, exact=exact)
    assert ok, f"worst |C - r| / tol = {worst} at {where}"


SHAPES = [
    (1, 1, 1 << 20),        # one dot product of 2^20 terms
    (16, 16, 1 << 20),      # few outputs, very long k
    (1 << 20, 16, 16),      # tall: 2^20 rows
    (16, 1 << 20, 16),      # wide: 2^20 columns
    (1 << 14, 1 << 10, 4),  # k below one slab
    (1, 4096, 4096),        # one row
    (4096, 1, 4096),        # one column
]


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
@pytest.mark.parametrize("m,n,k", SHAPES, ids=lambda v: str(v))
def test_extreme_shapes(path, m, n, k):
    p = inputs.make_problem(m, n, k, alpha=1.5, beta=0.5, seed=(m * 31 + n * 7 + k) % 1000, a="normal",
                            b="uniform", c="uniform")
    _run(p, path)


@pytest.mark.parametrize("path", [binding.PATH_TF32X3, binding.PATH_FFMA], ids=["tf32x3", "ffma"])
@pytest.mark.parametrize("m,n,k", [(1 << 20, 16, 16), (16, 1 << 20, 16), (64, 64, 1 << 18)], ids=lambda v: str(v))
def test_extreme_shapes_integer_twin_bit_exact(path, m, n, k):
    """Entries in {-4..4}: with k <= 2^18 every partial sum is an integer of
    magnitude below 16 * 2^18 < 2^24, so any summation order is exact."""
    p = inputs.make_problem(m, n, k, alpha=1.0, beta=0.0, seed=5, a="int", b="int")
    _run(p, path, exact=True)
