"""The allocation-free tensor-core entry point, sgemm_tf32x3_noalloc.

Some callers must not allocate device memory while they run: code inside an
allocator callback or an out-of-memory handler (an allocation there can
recurse or deadlock on the allocator's own lock), processes that reserve all
of their device memory up front and leave none to a library, and
latency-critical loops that cannot risk cudaMalloc's implicit
synchronisation or its failure under memory pressure.  The regular entry
point takes scratch from a stream-ordered pool when an operand cannot be
read by TMA as stored (rows not 16 bytes apart, a misaligned base) or when
its plan uses stream-K; this entry point instead puts the split operands in
one fixed 64 MiB device array and plans without stream-K.

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


# (m, n, k, seed, lda pad): odd pads make A's rows misaligned (A split into
# the fixed scratch), even ones leave A readable as stored
@pytest.mark.parametrize("shapes", [
    [(1000, 1500, 777, 2, 0), (300, 200, 150, 3, 1)],
    [(2048, 2048, 2048, 5, 1), (129, 257, 1000, 6, 0)],
])
def test_noalloc_matches_oracle_twice(shapes, monkeypatch):
    # the regular call is planned without stream-K, as this entry point is,
    # so that both run the same kernels
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "0")
    stream = torch.cuda.current_stream().cuda_stream
    for m, n, k, seed, pad in shapes:
        p = inputs.make_problem(m, n, k, alpha=1.5, beta=0.5, seed=seed, a="normal", b="uniform", c="uniform",
                                lda=k + pad)
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
    reports out-of-memory.  On a problem whose A must be split into scratch
    (lda = 777: rows not 16 bytes apart) the regular entry point then fails
    with status 100 and leaves C alone; the allocation-free one succeeds,
    twice in a row, and matches the oracle."""
    stream = torch.cuda.current_stream().cuda_stream
    p = inputs.workload("1000x1500x777")
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


@pytest.mark.parametrize("name", ["8192^3", "16384x128x8192"])
def test_noalloc_large_workloads_with_allocations_failing(name, monkeypatch):
    """The two large workloads need no scratch at all through this entry
    point (both operands read as stored: CTA pairs at 8192^3, transposed
    tiles at n = 128), so they run with every pool allocation made to fail;
    checked on 4096 sampled outputs plus every tile edge."""
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
    """Only operands that cannot be read as stored take scratch: 2 * rows *
    ka floats each (ka = k rounded up to 4).  With both operands' rows
    misaligned (lda = ldb = 2049), m = n = 2048 and k = 2048 fill the array
    exactly; k = 2049 (ka = 2052) does not fit and is rejected before
    anything is enqueued, while the same shape with 16-byte rows needs no
    scratch at all."""
    assert binding.NOALLOC_SCRATCH_FLOATS == 2 * (2048 + 2048) * 2048
    st = binding.tf32x3_noalloc_raw(2048, 2048, 2049, 1.0, 256, 2049, 512, 2049, 0.0, 1024, 2048, 0)
    assert st == 97
    assert "scratch" in binding.status_string(st)
    # a problem that fits exactly, and one that needs no scratch, both run
    stream = torch.cuda.current_stream().cuda_stream
    for k, ld in ((2048, 2049), (2049, 2052)):
        p = inputs.make_problem(2048, 2048, k, alpha=1.0, beta=0.0, seed=k, a="uniform", b="uniform",
                                lda=ld, ldb=ld)
        A, B, C = _device(p.A), _device(p.B), _device(p.C0)
        st = _noalloc(p, A, B, C, stream)
        assert st == 0, binding.status_string(st)
        torch.cuda.synchronize()
        rows, cols = inputs.sample_indices(p.m, p.n, 512, seed=k)
        R, E = oracle.problem_f64_sampled(p, rows, cols)
        ok, worst, _ = oracle.within_tolerance(C.cpu().numpy()[rows, cols], R, E, 0.0, None)
        assert ok, worst
