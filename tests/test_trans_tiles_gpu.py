"""GPU parity of the transposed tensor-core tiles (n <= 128: the kernel
computes 256 x 128 tiles of C^T = B^T A^T so that its MMA stays 256 wide),
pinned through the library's tuning variable SGEMM_GB300_TRANS, against
the FP64 oracle: ragged m and n, k tails, padded lda, beta != 0, split-K
clusters, the in-kernel A split on and off, integer twins bit-exact,
strided batches and transposed operands."""
import pytest
import torch

from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import Placed, check_full
from test_batched_gpu import run_batch
from test_transpose_gpu import run as run_op

pytestmark = pytest.mark.gpu

TC = binding.PATH_TF32X3


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(autouse=True)
def _trans(monkeypatch):
    monkeypatch.setenv("SGEMM_GB300_TRANS", "1")


@pytest.fixture(params=["1", "0"], ids=["a_in_kernel", "a_pre_pass"])
def a_split(request, monkeypatch):
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", request.param)
    return request.param == "1"


def _plan(p):
    st, plan = binding.plan(p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, path=TC, num_sms=0)
    assert st == 0
    return plan


def _run(p, exact=False):
    pl = Placed(p)
    st = pl.run(TC)
    assert st == 0, binding.status_string(st)
    C, guard_ok = pl.result()
    assert guard_ok, "a write landed outside the m x n window of C"
    assert pl.inputs_untouched(), "A or B was modified"
    ok, worst, where = check_full(p, C, exact=exact)
    assert ok, f"worst |C - r| / tol = {worst} at {where}"


@pytest.mark.parametrize("m,n,k,lda,beta", [
    (1000, 100, 777, 780, 0.5),      # ragged m (1000 = 3 x 256 + 232) and n, k % 16 = 9
    (4096, 128, 512, None, 0.0),     # full tiles
    (513, 128, 2048, None, -1.0),    # few tiles: split-K clusters
    (300, 1, 300, None, 0.0),        # one column
    (257, 127, 4096, 4100, 2.0),     # ragged, long k, padded lda
    (2048, 64, 1000, None, 0.0),     # n = 64: half of the 128-row operand is zero fill
])
def test_trans_tiles_match_oracle(a_split, m, n, k, lda, beta):
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=beta, seed=m + 3 * n + k, a="normal", b="uniform",
                            c="uniform" if beta else None, lda=lda)
    plan = _plan(p)
    assert plan["trans"] == 1 and (plan["bm"], plan["bn"]) == (256, 128), plan
    assert plan["a_in_kernel"] == int(a_split)
    _run(p)


@pytest.mark.parametrize("m,n,k", [(1000, 100, 777), (513, 128, 2048), (3000, 32, 4096)])
def test_trans_tiles_integer_twin_bit_exact(a_split, m, n, k):
    lda = (k + 3) // 4 * 4
    p = inputs.make_problem(m, n, k, alpha=2.0, beta=0.5, seed=5 * k + n, a="int", b="int", c="int", lda=lda)
    assert _plan(p)["trans"] == 1
    _run(p, exact=True)


def test_trans_tiles_split_k_forced(monkeypatch):
    """Every split-K factor on transposed tiles (the cluster reduction maps
    tile rows to columns of C)."""
    p = inputs.make_problem(700, 90, 3000, alpha=1.0, beta=0.5, seed=3, a="normal", b="normal", c="uniform",
                            lda=3000)
    for s in (2, 3, 5, 8):
        monkeypatch.setenv("SGEMM_GB300_SPLIT_K", str(s))
        plan = _plan(p)
        assert plan["trans"] == 1 and plan["split_k"] == s, plan
        _run(p)


@pytest.mark.parametrize("op_a,op_b", [(0, 1), (1, 0), (1, 1)], ids=["NT", "TN", "TT"])
def test_trans_tiles_transposed_operands(op_a, op_b):
    run_op(1000, 100, 777, op_a, op_b, TC, seed=21)


def test_trans_tiles_strided_batch():
    run_batch(3, 700, 96, 500, TC, seed=40)
    run_batch(4, 300, 128, 1200, TC, dist="int", exact=True, seed=41)


def test_plan_prefers_trans_for_the_skinny_workload(monkeypatch):
    monkeypatch.delenv("SGEMM_GB300_TRANS")
    st, plan = binding.plan(16384, 128, 8192, path=TC, num_sms=0)
    assert st == 0 and plan["trans"] == 1 and plan["grid"] >= 128, plan
