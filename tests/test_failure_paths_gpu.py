"""The failure-reporting paths, exercised without faulting, trapping or
hanging the GPU: (1) a bounded wait that runs out (a barrier nothing
signals, through the same bounded-wait routine as the GEMM's pipeline
waits) records its code in the device status word and the context stays
usable; (2) a forced allocation failure (host-side fake of the pool
allocation, SGEMM_GB300_FAIL_ALLOC) returns status 100 with the CUDA error
kept and C unwritten, and the next call succeeds."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_06_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

CUDA_ERROR_MEMORY_ALLOCATION = 2


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _gemm_matches_oracle(path=binding.PATH_TF32X3, seed=7):
    p = inputs.make_problem(300, 260, 500, alpha=1.5, beta=0.5, seed=seed, a="normal", b="uniform", c="uniform")
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C = torch.from_numpy(p.C0).cuda()
    binding.sgemm_ex(A, B, C, p.alpha, p.beta, path=path)
    R, E, _ = oracle.problem_f64(p)
    ok, worst, where = oracle.within_tolerance(C.cpu().numpy(), R, E, p.beta, p.C0)
    return ok, worst, where


def test_bounded_wait_runs_out_and_is_reported():
    binding.device_status(clear=True)
    assert binding.selftest_wait(2_000_000)          # 2 ms, nothing signals the barrier
    assert binding.device_status(clear=True) == 0x207
    assert binding.device_status() == 0
    # the context is still usable, and a real call leaves the word clear
    ok, worst, where = _gemm_matches_oracle()
    assert ok, f"after the self-test: |C - r| / tol = {worst} at {where}"
    assert binding.device_status() == 0


def test_forced_allocation_failure(monkeypatch):
    # ldb = 386: B's rows are not 16-byte aligned, so the tensor-core call
    # splits B into scratch from the pool -- the allocation the fake fails
    p = inputs.make_problem(512, 384, 256, alpha=1.0, beta=0.5, seed=11, a="uniform", b="uniform", c="uniform",
                            ldb=386)
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C = torch.from_numpy(p.C0).cuda()
    C0 = C.clone()
    monkeypatch.setenv("SGEMM_GB300_FAIL_ALLOC", "1")
    st = binding.sgemm_raw(p.m, p.n, p.k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta, C.data_ptr(),
                           p.ldc, torch.cuda.current_stream().cuda_stream, binding.PATH_TF32X3)
    assert st == 100 and binding.last_cuda_error() == CUDA_ERROR_MEMORY_ALLOCATION
    with pytest.raises(binding.SgemmError) as err:
        binding.sgemm_ex(A, B[:, :p.n], C, p.alpha, p.beta, path=binding.PATH_TF32X3)
    assert err.value.status == 100
    torch.cuda.synchronize()
    assert torch.equal(C, C0), "C was written although the call failed before launching"
    # the FFMA path allocates nothing and is unaffected
    binding.sgemm_ex(A, B[:, :p.n], C, p.alpha, p.beta, path=binding.PATH_FFMA)
    R, E, _ = oracle.problem_f64(p)
    ok, worst, _ = oracle.within_tolerance(C.cpu().numpy(), R, E, p.beta, p.C0)
    assert ok, worst
    monkeypatch.delenv("SGEMM_GB300_FAIL_ALLOC")
    C.copy_(C0)
    binding.sgemm_ex(A, B[:, :p.n], C, p.alpha, p.beta, path=binding.PATH_TF32X3)
    ok, worst, _ = oracle.within_tolerance(C.cpu().numpy(), R, E, p.beta, p.C0)
    assert ok, worst
    assert binding.device_status() == 0


@pytest.mark.parametrize("lda", [768, 769, 771])
def test_tensor_core_call_with_readable_b_allocates_nothing(lda, monkeypatch):
    """With B's rows 16 bytes apart the tensor-core GEMM reads B as stored,
    and A as stored too -- by TMA when its rows are 16 bytes apart, else
    (lda = 769, 771) in four row phases that TMA can read -- so the call takes
    no scratch: it succeeds while every pool allocation is made to fail, and
    matches the oracle."""
    p = inputs.make_problem(1024, 512, 768, alpha=1.5, beta=0.5, seed=12, a="normal", b="uniform", c="uniform",
                            lda=lda)
    st, plan = binding.plan(p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc,
                            path=binding.PATH_TF32X3)
    assert st == 0 and plan["a_in_kernel"] == 1 and plan["b_in_kernel"] == 1 and plan["stream_k"] == 0, plan
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C = torch.from_numpy(p.C0).cuda()
    monkeypatch.setenv("SGEMM_GB300_FAIL_ALLOC", "1")
    binding.sgemm_ex(A[:, :p.k], B, C, p.alpha, p.beta, path=binding.PATH_TF32X3)
    R, E, _ = oracle.problem_f64(p)
    ok, worst, _ = oracle.within_tolerance(C.cpu().numpy(), R, E, p.beta, p.C0)
    assert ok, worst
    assert binding.device_status() == 0
