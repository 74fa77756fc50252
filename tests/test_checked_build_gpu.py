"""The bounds-checking build (SGEMM_GB300_CHECKED, the second library that
build() makes): every kernel tests each global and shared-memory index it
computes against the buffer it addresses before the access, and a failed
test skips the access and records 0x208 with the test's source line.

Here every entry point runs through that library (the binding is pointed at
it for this module) on problems that reach each kernel and each of its
paths -- ragged tiles and k tails, padded and misaligned operands, an A read
in row phases, split-K clusters, stream-K, CTA pairs, transposed tiles, the
FFMA path's two tiles, transposed operands, strided batches, the split
entry points, the allocation-free entry point and the reduction -- and
each must match the FP64 oracle with no test failed.  A self-test makes one
test fail on purpose (on a store it then skips) to show that the checks are
compiled in and reported."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_06_gb300 import _native, binding, inputs
from test_batched_gpu import run_batch
from test_parity_gpu import run_and_check

pytestmark = pytest.mark.gpu

TC, FFMA = binding.PATH_TF32X3, binding.PATH_FFMA


@pytest.fixture(autouse=True, scope="module")
def checked_lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    lib = _native.load(checked=True)
    assert lib.sgemm_version().endswith(b"checked)")
    mp = pytest.MonkeyPatch()
    mp.setattr(_native, "load", lambda *a, **k: lib)
    yield lib
    mp.undo()


def bounds_line(lib, clear=False):
    line = ctypes.c_int(-1)
    assert lib.sgemm_bounds_line(ctypes.byref(line), int(clear)) == 0
    return line.value


@pytest.fixture(autouse=True)
def _no_failed_test(checked_lib, monkeypatch):
    for v in ("SGEMM_GB300_STREAM_K", "SGEMM_GB300_PAIR", "SGEMM_GB300_SPLIT_K", "SGEMM_GB300_TILE_N",
              "SGEMM_GB300_TRANS", "SGEMM_GB300_SPLIT_A_IN", "SGEMM_GB300_SPLIT_B_IN", "SGEMM_GB300_FFMA_RN"):
        monkeypatch.delenv(v, raising=False)
    binding.device_status(clear=True)
    yield
    line = bounds_line(checked_lib)
    assert binding.device_status() == 0 and line == 0, f"a bounds test failed at source line {line}"


def test_selftest_records_a_failed_test(checked_lib):
    line = ctypes.c_int(0)
    assert checked_lib.sgemm_selftest_bounds(ctypes.byref(line)) == 0
    assert line.value > 0
    assert binding.device_status(clear=True) == 0x208
    assert bounds_line(checked_lib) == 0


@pytest.mark.parametrize("path", [FFMA, TC], ids=["ffma", "tf32x3"])
@pytest.mark.parametrize("m,n,k,lda,ldb,ldc,offs", [
    (129, 257, 77, None, None, None, (0, 0, 0)),
    (1000, 1500, 777, 777, None, None, (0, 0, 0)),       # A in row phases, split-K clusters
    (300, 200, 150, 161, 203, 260, (0, 0, 0)),           # padded, misaligned rows of B
    (260, 140, 90, None, None, None, (3, 2, 1)),         # misaligned bases
    (129, 257, 4096, None, None, None, (0, 0, 0)),       # split-K over a long k
    (3000, 100, 2048, None, None, None, (0, 0, 0)),      # transposed tiles (n <= 128)
    (1, 1, 1, None, None, None, (0, 0, 0)),
])
def test_problems_pass_every_bounds_test(path, m, n, k, lda, ldb, ldc, offs):
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=0.5, seed=m + n + k, a="normal", b="uniform", c="uniform",
                            lda=lda, ldb=ldb, ldc=ldc)
    run_and_check(p, path, offs=offs)


@pytest.mark.parametrize("env,m,n,k", [
    ({"SGEMM_GB300_STREAM_K": "1"}, 3000, 2000, 999),                    # stream-K, A in row phases
    ({"SGEMM_GB300_STREAM_K": "1"}, 16384, 128, 1024),                   # stream-K on transposed tiles
    ({"SGEMM_GB300_PAIR": "1", "SGEMM_GB300_SPLIT_B_IN": "1"}, 700, 600, 1000),   # CTA pairs
    ({"SGEMM_GB300_TILE_N": "128", "SGEMM_GB300_SPLIT_K": "3"}, 300, 500, 777),   # 128-wide tiles, split-K 3
    ({"SGEMM_GB300_SPLIT_A_IN": "0", "SGEMM_GB300_SPLIT_B_IN": "0"}, 500, 300, 333),  # both split first
])
def test_pinned_plans_pass_every_bounds_test(monkeypatch, env, m, n, k):
    for key, val in env.items():
        monkeypatch.setenv(key, val)
    p = inputs.make_problem(m, n, k, alpha=0.75, beta=1.0, seed=k, a="normal", b="uniform", c="uniform")
    run_and_check(p, TC)


def test_ffma_8x16(monkeypatch):
    monkeypatch.setenv("SGEMM_GB300_FFMA_RN", "16")
    p = inputs.make_problem(300, 600, 70, alpha=1.0, beta=-1.0, seed=31, a="uniform", b="normal", c="normal")
    run_and_check(p, FFMA)


@pytest.mark.parametrize("path", [FFMA, TC], ids=["ffma", "tf32x3"])
@pytest.mark.parametrize("op_a,op_b", [(0, 1), (1, 0), (1, 1)])
def test_transposed_operands(path, op_a, op_b):
    m, n, k = 200, 260, 130
    rng = np.random.default_rng(7 + 2 * op_a + op_b)
    A = rng.standard_normal((k, m) if op_a else (m, k)).astype(np.float32)
    B = rng.uniform(-1, 1, (n, k) if op_b else (k, n)).astype(np.float32)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.zeros(m, n, device="cuda")
    st = binding.sgemm_op_raw(op_a, op_b, m, n, k, 1.0, Ad.data_ptr(), A.shape[1], Bd.data_ptr(), B.shape[1], 0.0,
                              C.data_ptr(), n, torch.cuda.current_stream().cuda_stream, path)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    R, E, _ = oracle.sgemm_f64(m, n, k, 1.0, np.ascontiguousarray(A.T if op_a else A), k,
                               np.ascontiguousarray(B.T if op_b else B), n, 0.0, None, n)
    ok, worst, where = oracle.within_tolerance(C.cpu().numpy(), R, E, 0.0, None)
    assert ok, (worst, where)


@pytest.mark.parametrize("path", [FFMA, TC], ids=["ffma", "tf32x3"])
def test_strided_batch(path):
    run_batch(3, 130, 257, 77, path, seed=17)


def test_split_entry_points_and_no_allocation():
    p = inputs.make_problem(300, 200, 150, alpha=1.5, beta=0.5, seed=5, a="normal", b="uniform", c="uniform",
                            lda=151, ldb=203)
    A, B = torch.from_numpy(p.A).cuda(), torch.from_numpy(p.B).cuda()
    C = torch.from_numpy(p.C0).cuda()
    st = binding.tf32x3_noalloc_raw(p.m, p.n, p.k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                                    C.data_ptr(), p.ldc, torch.cuda.current_stream().cuda_stream)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    R, E, _ = oracle.problem_f64(p)
    ok, worst, _ = oracle.within_tolerance(C.cpu().numpy(), R, E, p.beta, p.C0)
    assert ok, worst
    ka = binding.ka_of(p.k)
    a_hi, a_lo = torch.empty(p.m * ka, device="cuda"), torch.empty(p.m * ka, device="cuda")
    b_hi, b_lo = torch.empty(p.n * ka, device="cuda"), torch.empty(p.n * ka, device="cuda")
    binding.tf32x3_split_a(A[:, :p.k], a_hi, a_lo)
    binding.tf32x3_split_b(B[:, :p.n], b_hi, b_lo)
    C2 = torch.from_numpy(p.C0).cuda()
    st = binding.tf32x3_split_gemm_raw(p.m, p.n, p.k, p.alpha, a_hi.data_ptr(), a_lo.data_ptr(), b_hi.data_ptr(),
                                       b_lo.data_ptr(), p.beta, C2.data_ptr(), p.ldc,
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    ok, worst, _ = oracle.within_tolerance(C2.cpu().numpy(), R, E, p.beta, p.C0)
    assert ok, worst


@pytest.mark.parametrize("n,off", [(1_000_003, 1), (4096, 0), (5, 3)])
def test_reduction(n, off):
    x = torch.empty(n + off, device="cuda").uniform_(-1, 1)
    out = torch.empty(1, device="cuda")
    st = binding.reduce_sum_raw(x.data_ptr() + 4 * off, n, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    ref = x[off:].double().sum().item()
    assert abs(out.item() - ref) <= 1e-5 * x[off:].double().abs().sum().item() + 1e-6
