"""GPU parity of the transposed forms C = alpha * op(A) * op(B) + beta * C
(SGEMM_OP_N / SGEMM_OP_T for each operand, row-major storage), both kernel
paths, against the FP64 oracle fed the logical op(A), op(B)."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import SENTINEL

pytestmark = pytest.mark.gpu

PATHS = {"ffma": binding.PATH_FFMA, "tf32x3": binding.PATH_TF32X3}
OPS = [(0, 0), (0, 1), (1, 0), (1, 1)]


def stored(x, op, ld_pad, seed):
    """The storage of logical matrix x for `op`: x itself (op N) or x^T
    (op T), row-major with ld = cols + ld_pad (padding NaN)."""
    s = x if op == 0 else np.ascontiguousarray(x.T)
    ld = s.shape[1] + ld_pad
    out = np.full((s.shape[0], ld), np.nan, dtype=np.float32)
    out[:, :s.shape[1]] = s
    return out, ld


def run(m, n, k, op_a, op_b, path, *, alpha=1.25, beta=0.5, dist="normal", pad=(0, 0), off=(0, 0), seed=0,
        exact=False):
    p = inputs.make_problem(m, n, k, alpha=alpha, beta=beta, seed=seed, a=dist, b=dist if dist != "normal" else "uniform",
                            c="int" if dist == "int" else "uniform")
    a_log = p.A[:, :k]
    b_log = p.B[:, :n]
    A_st, lda = stored(a_log, op_a, pad[0], seed)
    B_st, ldb = stored(b_log, op_b, pad[1], seed)

    def dev(arr, o):
        flat = np.concatenate([np.full(o, SENTINEL, np.float32), arr.reshape(-1)])
        t = torch.from_numpy(flat).cuda()
        return t, t.data_ptr() + 4 * o

    tA, pA = dev(A_st, off[0])
    tB, pB = dev(B_st, off[1])
    C = torch.from_numpy(p.C0).cuda()
    st = binding.sgemm_op_raw(op_a, op_b, m, n, k, p.alpha, pA, lda, pB, ldb, p.beta, C.data_ptr(), p.ldc,
                              torch.cuda.current_stream().cuda_stream, path)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    got = C.cpu().numpy()[:, :n]
    R, E, Rf = oracle.sgemm_f64(m, n, k, p.alpha, a_log, k, b_log, n, p.beta, p.C0[:, :n], n)
    if exact:
        assert np.array_equal(got, Rf)
    else:
        ok, worst, where = oracle.within_tolerance(got, R, E, p.beta, p.C0[:, :n])
        assert ok, f"worst {worst} at {where}"


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
@pytest.mark.parametrize("op_a,op_b", OPS, ids=["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("m,n,k", [(300, 260, 150), (129, 257, 33), (5, 7, 3), (1000, 1500, 777), (64, 64, 4096)])
def test_transposes(m, n, k, op_a, op_b, path):
    run(m, n, k, op_a, op_b, path, seed=m + 3 * n + 7 * k + op_a + 2 * op_b)


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
@pytest.mark.parametrize("op_a,op_b", OPS, ids=["NN", "NT", "TN", "TT"])
def test_transposes_integer_twin_bit_exact(op_a, op_b, path):
    run(257, 301, 190, op_a, op_b, path, alpha=2.0, beta=0.5, dist="int", seed=5 + op_a + 2 * op_b, exact=True)


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
@pytest.mark.parametrize("op_a,op_b", OPS, ids=["NN", "NT", "TN", "TT"])
def test_transposes_padded_and_misaligned(op_a, op_b, path):
    run(200, 180, 140, op_a, op_b, path, pad=(3, 5), off=(1, 3), seed=77 + op_a + 2 * op_b)


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
def test_matmul_on_transposed_views(path):
    torch.manual_seed(3)
    X = torch.randn(96, 130, device="cuda")    # A = X^T: 130 x 96
    Y = torch.randn(70, 96, device="cuda")     # B = Y^T: 96 x 70
    C = torch.zeros(130, 70, device="cuda")
    binding.matmul(X.t(), Y.t(), C, path=path)
    ref = X.t().double() @ Y.t().double()
    E = X.t().double().abs() @ Y.t().double().abs()
    assert torch.all((C.double() - ref).abs() <= 1e-5 * E)
