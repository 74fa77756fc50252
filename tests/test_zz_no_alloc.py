"""The allocation-free tensor-core entry point, sgemm_tf32x3_noalloc.

Some callers must not allocate device memory while they run: code inside an
allocator callback or an out-of-memory handler (an allocation there can
recurse or deadlock on the allocator's own lock), processes that reserve all
of their device memory up front and leave none to a library, and
latency-critical loops that cannot risk cudaMalloc's implicit
synchronisation or its failure under memory pressure.  The regular entry
point takes scratch from a stream-ordered pool when B cannot be read by TMA
as stored (rows not 16 bytes apart, a misaligned base), when a plan splits
a large B first, or when its plan uses stream-K; this entry point reads
every operand it can as stored (an A that TMA cannot read as one tensor is
read in four row phases), puts a misaligned B's split parts in one fixed
64 MiB device array, and plans without stream-K.

These tests call it through the C ABI and hold its output to the FP64
oracle within the bound every parity test uses, twice in a row (the second
time on a smaller problem, so that whatever the first call left in the
shared array must not leak into the second result), with the regular entry
point's result as a second reference.  They also check the property the
entry point exists for: with every pool allocation made to fail, it still
succeeds while the regular entry point on the same problem reports the
failed allocation.

This file is collected last on purpose: if it fails, a run that stops at
the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_06_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _device(arr):
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def _noalloc(p, A, B, C, stream):
    return binding.tf32x3_noalloc_raw(p.m, p.n, p.k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                                      C.data_ptr(), p.ldc, stream)


def _regular(p, A, B, C, stream):
    return binding.sgemm_raw(p.m, p.n, p.k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                             C.data_ptr(), p.ldc, stream, binding.PATH_TF32X3)


def _check_oracle(p, got):
    R, E, _ = oracle.problem_f64(p)
    ok, worst, where = oracle.within_tolerance(got, R, E, p.beta, p.C0[:, :p.n])
    assert ok, f"|C - r| / tol = {worst} at {where}"
    return R, E


# (m, n, k, seed, lda pad, ldb pad): odd lda pads make A's rows misaligned
# (A read in row phases), ldb pads that are not multiples of 4 B's (B split
# into the fixed scratch)
@pytest.mark.parametrize("shapes", [
    [(1000, 1500, 777, 2, 0, 0), (300, 200, 150, 3, 1, 2)],
    [(2048, 2048, 2048, 5, 1, 0), (129, 257, 1000, 6, 0, 3)],
    [(700, 900, 500, 7, 3, 1), (2048, 2048, 2048, 8, 0, 0)],
])
def test_noalloc_matches_oracle_twice(shapes, monkeypatch):
    # the regular call is planned without stream-K, as this entry point is,
    # so that both run the same kernels where their plans agree
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "0")
    stream = torch.cuda.current_stream().cuda_stream
    for m, n, k, seed, pad_a, pad_b in shapes:
        p = inputs.make_problem(m, n, k, alpha=1.5, beta=0.5, seed=seed, a="normal", b="uniform", c="uniform",
                                lda=k + pad_a, ldb=n + pad_b)
        A, B = _device(p.A), _device(p.B)
        C_na, C_ref = _device(p.C0), _device(p.C0)
        st = _noalloc(p, A, B, C_na, stream)
        assert st == 0, binding.status_string(st)
        st = _regular(p, A, B, C_ref, stream)
        assert st == 0, binding.status_string(st)
        torch.cuda.synchronize()
        got = C_na.cpu().numpy()[:, :p.n]
        assert np.all(np.isfinite(got))
        R, E = _check_oracle(p, got)
        # the regular entry point's result, within the same bound of it
        ref = C_ref.cpu().numpy()[:, :p.n].astype(np.float64)
        assert np.all(np.abs(got - ref) <= oracle.tolerance(E, p.beta, p.C0[:, :p.n]))


def test_noalloc_needs_no_allocation(monkeypatch):
    """With SGEMM_GB300_FAIL_ALLOC set every pool allocation of the library
    reports out-of-memory.  On a problem whose B must be split into scratch
    (ldb = 1501: rows not 16 bytes apart; A's rows misaligned too, lda = 777)
    the regular entry point then fails with status 100 and leaves C alone;
    the allocation-free one succeeds, twice in a row, and matches the
    oracle."""
    stream = torch.cuda.current_stream().cuda_stream
    p = inputs.make_problem(1000, 1500, 777, alpha=1.5, beta=0.5, seed=2, a="uniform", b="uniform", c="normal",
                            ldb=1501)
    assert p.lda == 777
    A, B = _device(p.A), _device(p.B)
    monkeypatch.setenv("SGEMM_GB300_FAIL_ALLOC", "1")
    C_ref = _device(p.C0)
    assert _regular(p, A, B, C_ref, stream) == 100
    for _ in range(2):
        C = _device(p.C0)
        st = _noalloc(p, A, B, C, stream)
        assert st == 0, binding.status_string(st)
        torch.cuda.synchronize()
        _check_oracle(p, C.cpu().numpy())
    assert np.array_equal(C_ref.cpu().numpy(), p.C0, equal_nan=True)


@pytest.mark.parametrize("name", ["1000x1500x777", "8192^3", "16384x128x8192"])
def test_noalloc_workloads_with_allocations_failing(name, monkeypatch):
    """The workloads need no scratch at all through this entry point (both
    operands read as stored: A in row phases at lda = 777, CTA pairs at
    8192^3, transposed tiles at n = 128), so they run with every pool
    allocation made to fail; checked on 4096 sampled outputs plus every tile
    edge."""
    monkeypatch.setenv("SGEMM_GB300_FAIL_ALLOC", "1")
    stream = torch.cuda.current_stream().cuda_stream
    p = inputs.workload(name)
    A, B, C = _device(p.A), _device(p.B), _device(p.C0)
    st = _noalloc(p, A, B, C, stream)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    rows, cols = inputs.sample_indices(p.m, p.n, 4096, seed=p.seed + 1000)
    R, E = oracle.problem_f64_sampled(p, rows, cols)
    got = C.cpu().numpy()[rows, cols]
    ok, worst, where = oracle.within_tolerance(got, R, E, p.beta, p.C0[rows, cols] if p.beta else None)
    assert ok, (worst, where)
    assert binding.device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Only a B that TMA cannot read takes scratch: 2 * n * ka floats (ka = k
    rounded up to 4).  With B's rows misaligned (ldb = 4097), n = 4096 and
    k = 2048 fill the array exactly; k = 2049 (ka = 2052) does not fit and is
    rejected before anything is enqueued, while the same shape with 16-byte
    rows needs no scratch at all."""
    assert binding.NOALLOC_SCRATCH_FLOATS == 2 * 4096 * 2048
    st = binding.tf32x3_noalloc_raw(512, 4096, 2049, 1.0, 256, 2049, 512, 4097, 0.0, 1024, 4096, 0)
    assert st == 97
    assert "scratch" in binding.status_string(st)
    # a problem that fits exactly, and one that needs no scratch, both run
    stream = torch.cuda.current_stream().cuda_stream
    for k, ldb in ((2048, 4097), (2049, 4100)):
        p = inputs.make_problem(512, 4096, k, alpha=1.0, beta=0.0, seed=k, a="uniform", b="uniform", ldb=ldb)
        A, B, C = _device(p.A), _device(p.B), _device(p.C0)
        st = _noalloc(p, A, B, C, stream)
        assert st == 0, binding.status_string(st)
        torch.cuda.synchronize()
        rows, cols = inputs.sample_indices(p.m, p.n, 512, seed=k)
        R, E = oracle.problem_f64_sampled(p, rows, cols)
        ok, worst, _ = oracle.within_tolerance(C.cpu().numpy()[rows, cols], R, E, 0.0, None)
        assert ok, worst
