"""GPU parity of the FFMA path's 8 x 16 outputs per thread (128-thread CTAs
of 128 x 128 tiles, two per SM), which the library takes from one wave of
such CTAs on and which SGEMM_GB300_FFMA_RN=16 pins here on small shapes:
ragged edges, padded and misaligned operands, transposed operands, strided
batches and integer twins against the FP64 oracle; and, because both FFMA
configurations sum every output in increasing k with one fmaf per product,
bit-identical results to the 8 x 8 configuration on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_06_gb300 import binding, inputs
from test_parity_gpu import run_and_check

pytestmark = pytest.mark.gpu

FFMA = binding.PATH_FFMA


@pytest.fixture(autouse=True)
def _deep(monkeypatch):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    monkeypatch.setenv("SGEMM_GB300_FFMA_RN", "16")


def test_pinned_plan_is_8x16():
    st, p = binding.plan(300, 500, 70, path=FFMA)
    assert st == 0 and (p["bm"], p["bn"], p["rm"], p["rn"], p["threads"]) == (128, 128, 8, 16, 128)
    assert p["tiles"] == 3 * 4 and p["grid"] == 12


@pytest.mark.parametrize("m,n,k", [
    (1, 1, 1), (1, 257, 5), (129, 1, 3), (127, 256, 129), (128, 256, 128), (129, 257, 129),
    (200, 31, 1), (5, 600, 300), (255, 513, 33), (385, 130, 47), (640, 768, 512),
])
def test_ragged_shapes(m, n, k):
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=-0.75, seed=m * 5 + n * 13 + k, c="uniform")
    run_and_check(p, FFMA)


def test_ragged_integer_sweep_bit_exact():
    rng = np.random.default_rng(77)
    edge = [1, 3, 4, 5, 127, 128, 129, 255, 256, 257, 300]
    for trial in range(12):
        m, n, k = (int(rng.choice(edge)) for _ in range(3))
        p = inputs.make_problem(m, n, k, alpha=2.0, beta=0.5, seed=900 + trial, a="int", b="int", c="int")
        run_and_check(p, FFMA, exact=True)


def test_padded_leading_dimensions():
    p = inputs.make_problem(300, 400, 150, alpha=1.0, beta=1.0, seed=19, c="uniform", lda=161, ldb=403, ldc=460)
    run_and_check(p, FFMA)


@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1)])
def test_misaligned_pointers(offs):
    p = inputs.make_problem(260, 300, 90, alpha=0.5, beta=2.0, seed=20, c="normal")
    run_and_check(p, FFMA, offs=offs)


@pytest.mark.parametrize("op_a,op_b", [(0, 1), (1, 0), (1, 1)])
def test_transposed_operands(op_a, op_b):
    m, n, k = 300, 520, 170
    rng = np.random.default_rng(op_a * 2 + op_b + 40)
    A = rng.standard_normal((k, m) if op_a else (m, k)).astype(np.float32)
    B = rng.uniform(-1, 1, (n, k) if op_b else (k, n)).astype(np.float32)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.zeros(m, n, device="cuda")
    st = binding.sgemm_op_raw(op_a, op_b, m, n, k, 1.0, Ad.data_ptr(), A.shape[1], Bd.data_ptr(), B.shape[1], 0.0,
                              C.data_ptr(), n, torch.cuda.current_stream().cuda_stream, FFMA)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    opA = A.T if op_a else A
    opB = B.T if op_b else B
    R, E, _ = oracle.sgemm_f64(m, n, k, 1.0, np.ascontiguousarray(opA), k, np.ascontiguousarray(opB), n, 0.0, None, n)
    ok, worst, where = oracle.within_tolerance(C.cpu().numpy(), R, E, 0.0, None)
    assert ok, (worst, where)


def test_strided_batch():
    batch, m, n, k = 3, 200, 300, 77
    rng = np.random.default_rng(41)
    A = rng.standard_normal((batch, m, k)).astype(np.float32)
    B = rng.uniform(-1, 1, (batch, k, n)).astype(np.float32)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.zeros(batch, m, n, device="cuda")
    st = binding.sgemm_strided_batched_raw(0, 0, m, n, k, 1.0, Ad.data_ptr(), k, m * k, Bd.data_ptr(), n, k * n, 0.0,
                                           C.data_ptr(), n, m * n, batch, torch.cuda.current_stream().cuda_stream, FFMA)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    for b in range(batch):
        R, E, _ = oracle.sgemm_f64(m, n, k, 1.0, A[b], k, B[b], n, 0.0, None, n)
        ok, worst, where = oracle.within_tolerance(got[b], R, E, 0.0, None)
        assert ok, (b, worst, where)


@pytest.mark.parametrize("m,n,k", [(1000, 1500, 777), (384, 1024, 2048)])
def test_same_bits_as_8x8(monkeypatch, m, n, k):
    p = inputs.make_problem(m, n, k, alpha=1.5, beta=0.5, seed=k, a="normal", b="uniform", c="uniform")
    A, B = torch.from_numpy(p.A).cuda(), torch.from_numpy(p.B).cuda()
    outs = []
    for rn in ("16", "8"):
        monkeypatch.setenv("SGEMM_GB300_FFMA_RN", rn)
        C = torch.from_numpy(p.C0).cuda()
        st = binding.sgemm_raw(p.m, p.n, p.k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta, C.data_ptr(),
                               p.ldc, torch.cuda.current_stream().cuda_stream, FFMA)
        assert st == 0, binding.status_string(st)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
