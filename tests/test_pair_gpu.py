"""GPU parity of the CTA-pair tensor-core GEMM (tcgen05 cta_group::2: two
CTAs of a cluster compute one 256 x 256 tile with M = 256 MMAs issued by
the even CTA, each CTA staging and splitting its 128 rows of A and its 128
rows of B), requested with the tuning variable SGEMM_GB300_PAIR, against
the FP64 oracle: exact identity products that name the element read at
every output (which half of each operand sits in which CTA), ragged
shapes, beta != 0, padded leading dimensions, transposed operands read
MN-major, strided batches, integer twins bit for bit, and repeatability."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import Placed, check_full

pytestmark = pytest.mark.gpu

TC = binding.PATH_TF32X3


@pytest.fixture(autouse=True)
def _pair(monkeypatch):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    for v in ("SGEMM_GB300_SPLIT_A_IN", "SGEMM_GB300_SPLIT_B_IN", "SGEMM_GB300_TRANS", "SGEMM_GB300_STREAM_K",
              "SGEMM_GB300_SPLIT_K", "SGEMM_GB300_TILE_N"):
        monkeypatch.delenv(v, raising=False)
    monkeypatch.setenv("SGEMM_GB300_PAIR", "1")


def _plan(m, n, k, lda=None, ldb=None):
    st, plan = binding.plan(m, n, k, 1.0, 256, lda or k, 256, ldb or n, 0.0, 256, n, path=TC)
    assert st == 0
    return plan


@pytest.mark.parametrize("m,n,k", [(256, 256, 256), (512, 768, 384), (300, 500, 200)])
def test_pair_identity_names_every_element(m, n, k):
    """C = I * X with X[t][j] = t + 256 (j % 256): every output is one exact
    product, so a half of A or B placed in the wrong CTA, or read in the
    wrong order, shows as the wrong value."""
    plan = _plan(m, n, k)
    assert plan["pair"] == 1 and plan["bm"] == 256 and plan["bn"] == 256 and plan["grid"] == 2 * plan["tiles"]
    t = np.arange(k, dtype=np.float64)[:, None]
    X = (t + 256.0 * (np.arange(n)[None, :] % 256)).astype(np.float32)
    A = np.eye(m, k, dtype=np.float32)
    want = np.zeros((m, n), np.float32)
    want[:min(m, k)] = X[:min(m, k)]
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(X).cuda()
    C = torch.full((m, n), -1.0, device="cuda")
    st = binding.sgemm_raw(m, n, k, 1.0, Ad.data_ptr(), k, Bd.data_ptr(), n, 0.0, C.data_ptr(), n,
                           torch.cuda.current_stream().cuda_stream, TC)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, [(int(i), int(j), float(got[i, j]), float(want[i, j])) for i, j in bad[:8]]
    assert binding.device_status() == 0


@pytest.mark.parametrize("m,n,k,lda,ldb,beta", [
    (256, 256, 1024, None, None, 0.0),    # one pair tile, long k
    (1000, 1500, 780, None, None, 0.5),    # ragged m and n, k % 16 = 12, beta
    (2048, 2048, 512, None, None, -1.0),   # 64 pair tiles
    (700, 600, 1000, 1004, 604, 2.0),      # padded leading dimensions
    (129, 257, 4096, 4096, 260, 0.0),      # one partial pair tile, long k
])
def test_pair_matches_oracle(m, n, k, lda, ldb, beta):
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=beta, seed=m + 3 * n + k, a="normal", b="uniform",
                            c="uniform" if beta else None, lda=lda, ldb=ldb)
    assert _plan(m, n, k, p.lda, p.ldb)["pair"] == 1
    pl = Placed(p)
    st = pl.run(TC)
    assert st == 0, binding.status_string(st)
    C, guard_ok = pl.result()
    assert guard_ok, "a write landed outside the m x n window of C"
    assert pl.inputs_untouched()
    ok, worst, where = check_full(p, C)
    assert ok, f"worst |C - r| / tol = {worst} at {where}"
    assert binding.device_status() == 0


@pytest.mark.parametrize("m,n,k", [(512, 512, 2048), (1000, 300, 777)])
def test_pair_integer_twin_bit_exact(m, n, k):
    lda, ldb = (k + 3) // 4 * 4, (n + 3) // 4 * 4
    p = inputs.make_problem(m, n, k, alpha=2.0, beta=0.5, seed=k + n, a="int", b="int", c="int", lda=lda,
                            ldb=ldb)
    assert _plan(m, n, k, lda, ldb)["pair"] == 1
    pl = Placed(p)
    assert pl.run(TC) == 0
    C, guard_ok = pl.result()
    assert guard_ok
    ok, _, where = check_full(p, C, exact=True)
    assert ok, where


@pytest.mark.parametrize("op_a,op_b", [(0, 1), (1, 0), (1, 1)])
def test_pair_transposed_operands(op_a, op_b):
    """op(A) = A^T is read MN-major (A stored k x m), op(B) = B^T K-major
    (B stored n x k)."""
    m, n, k = 640, 520, 700
    rng = np.random.default_rng(op_a * 2 + op_b)
    A = rng.standard_normal((k, m) if op_a else (m, k)).astype(np.float32)
    B = rng.uniform(-1, 1, (n, k) if op_b else (k, n)).astype(np.float32)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.zeros(m, n, device="cuda")
    st = binding.sgemm_op_raw(op_a, op_b, m, n, k, 1.0, Ad.data_ptr(), A.shape[1], Bd.data_ptr(), B.shape[1], 0.0,
                              C.data_ptr(), n, torch.cuda.current_stream().cuda_stream, TC)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    opA = A.T if op_a else A
    opB = B.T if op_b else B
    R, E, _ = oracle.sgemm_f64(m, n, k, 1.0, np.ascontiguousarray(opA), k, np.ascontiguousarray(opB), n, 0.0, None, n)
    ok, worst, where = oracle.within_tolerance(C.cpu().numpy(), R, E, 0.0, None)
    assert ok, (worst, where)


def test_pair_strided_batch():
    """Three problems in one launch (grid y = problem), B shared (stride 0)."""
    batch, m, n, k = 3, 300, 400, 500
    rng = np.random.default_rng(5)
    A = rng.standard_normal((batch, m, k)).astype(np.float32)
    B = rng.uniform(-1, 1, (k, n)).astype(np.float32)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.zeros(batch, m, n, device="cuda")
    st = binding.sgemm_strided_batched_raw(0, 0, m, n, k, 1.0, Ad.data_ptr(), k, m * k, Bd.data_ptr(), n, 0, 0.0,
                                           C.data_ptr(), n, m * n, batch, torch.cuda.current_stream().cuda_stream, TC)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    for b in range(batch):
        R, E, _ = oracle.sgemm_f64(m, n, k, 1.0, A[b], k, B, n, 0.0, None, n)
        ok, worst, where = oracle.within_tolerance(got[b], R, E, 0.0, None)
        assert ok, (b, worst, where)


def test_pair_is_repeatable():
    p = inputs.make_problem(1024, 1024, 1536, alpha=1.0, beta=0.0, seed=9, a="normal", b="normal")
    A, B = torch.from_numpy(p.A).cuda(), torch.from_numpy(p.B).cuda()
    outs = []
    for _ in range(3):
        C = torch.zeros(p.m, p.n, device="cuda")
        binding.sgemm_ex(A, B, C, 1.0, 0.0, path=TC)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
