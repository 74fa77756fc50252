"""The allocation-free tensor-core entry point, sgemm_tf32x3_noalloc.

Some callers must not allocate device memory while they run (allocator
callbacks, out-of-memory handlers, processes that reserve all device memory
up front, latency-critical loops that cannot risk cudaMalloc's
synchronisation or failure).  For them the library offers one entry point
whose scratch is a fixed 64 MiB device array instead of the stream-ordered
pool.  These tests call it through the C ABI and hold its output to the
same bound as every other parity test, against the regular entry point
(sgemm_ex with the tensor-core path) on the same inputs -- twice in a row,
the second time on a smaller problem, so that whatever the first call left
in the shared array must not leak into the second result.

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


@pytest.mark.parametrize("shapes", [
    [(1000, 1500, 777, 2), (300, 200, 150, 3)],
    [(2048, 2048, 2048, 5), (129, 257, 1000, 6)],
])
def test_noalloc_matches_regular_entry_point_twice(shapes, monkeypatch):
    # the no-allocation entry point splits A with the pre-pass and runs
    # without stream-K (no workspace); the regular call is pinned to the
    # same (it may otherwise split A inside the GEMM, which rounds hi
    # differently, or add stream-K partial tiles in another order) so both
    # run the same kernels
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", "0")
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "0")
    stream = torch.cuda.current_stream().cuda_stream
    for m, n, k, seed in shapes:
        p = inputs.make_problem(m, n, k, alpha=1.5, beta=0.5, seed=seed, a="normal", b="uniform", c="uniform",
                                lda=k + (1 if seed % 2 else 0))
        A, B = _device(p.A), _device(p.B)
        C_ref, C_na = _device(p.C0), _device(p.C0)
        st = binding.sgemm_raw(m, n, k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                               C_ref.data_ptr(), p.ldc, stream, binding.PATH_TF32X3)
        assert st == 0, binding.status_string(st)
        st = binding.tf32x3_noalloc_raw(m, n, k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                                        C_na.data_ptr(), p.ldc, stream)
        assert st == 0, binding.status_string(st)
        torch.cuda.synchronize()
        ref = C_ref.cpu().numpy()[:, :n].astype(np.float64)
        got = C_na.cpu().numpy()[:, :n].astype(np.float64)
        # the bound of every parity test, with the regular entry point's result
        # standing in for r; E from the oracle's error scale
        _, E, _ = oracle.problem_f64(p)
        bound = oracle.tolerance(E, p.beta, p.C0[:, :n])
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - ref) <= bound)
        # same kernels on the same operands: in practice bit-identical
        assert np.array_equal(got, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 2 * (m + n) * ka floats are needed; 2048^3 fills the array exactly,
    # one more row does not fit.  Rejected before anything is enqueued.
    assert binding.NOALLOC_SCRATCH_FLOATS == 2 * (2048 + 2048) * 2048
    st = binding.tf32x3_noalloc_raw(2049, 2048, 2048, 1.0, 256, 2048, 512, 2048, 0.0, 1024, 2048, 0)
    assert st == 97
    assert "scratch" in binding.status_string(st)
