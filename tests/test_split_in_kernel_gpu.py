"""GPU parity of the tensor-core path with A split inside the GEMM kernel
(raw FP32 A loaded by TMA and read as its own hi part, lo computed in
shared memory) and with A split by the separate pre-pass, each pinned
through the library's tuning variable SGEMM_GB300_SPLIT_A_IN and checked
against the FP64 oracle:
ragged tiles, k tails that are not a multiple of the 16-deep slab, split-K
clusters, beta != 0, padded lda, and bit-exact integer twins."""
import pytest
import torch

from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import Placed, check_full

pytestmark = pytest.mark.gpu

TC = binding.PATH_TF32X3


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(params=["1", "0"], ids=["in_kernel", "pre_pass"])
def a_split(request, monkeypatch):
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", request.param)
    return request.param == "1"


def _run(p, exact=False):
    pl = Placed(p)
    st = pl.run(TC)
    assert st == 0, binding.status_string(st)
    C, guard_ok = pl.result()
    assert guard_ok, "a write landed outside the m x n window of C"
    assert pl.inputs_untouched(), "A or B was modified"
    ok, worst, where = check_full(p, C, exact=exact)
    assert ok, f"worst |C - r| / tol = {worst} at {where}"


def _plan(p):
    st, plan = binding.plan(p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, path=TC, num_sms=0)
    assert st == 0
    return plan


@pytest.mark.parametrize("m,n,k,lda,beta", [
    (256, 128, 4096, None, 0.0),     # one tile column, long k
    (1000, 300, 777, 780, 0.5),      # ragged m and n, k % 16 = 9, padded lda
    (129, 257, 4096, None, -1.0),    # split-K clusters (few tiles)
    (300, 700, 5000, 5004, 0.75),    # split-K, ragged, padded lda
    (2048, 64, 1000, None, 0.0),     # n below one narrow tile
    (640, 1024, 2048, None, 2.0),    # wide tiles
    (128, 128, 4, None, 0.0),        # one slab, k = 4
])
def test_in_kernel_and_pre_pass_split_match_oracle(a_split, m, n, k, lda, beta):
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=beta, seed=m * 7 + n + k, a="normal", b="uniform",
                            c="uniform" if beta else None, lda=lda)
    plan = _plan(p)
    assert plan["a_in_kernel"] == int(a_split), plan
    assert plan["threads"] == (384 if a_split else 320), plan
    _run(p)


@pytest.mark.parametrize("m,n,k", [(1000, 300, 777), (129, 257, 4096), (512, 512, 2048)])
def test_in_kernel_split_integer_twin_bit_exact(a_split, m, n, k):
    """hi(x) = x and lo(x) = 0 for small integers, so every product and
    partial sum is exact whichever side splits A."""
    lda = (k + 3) // 4 * 4
    p = inputs.make_problem(m, n, k, alpha=2.0, beta=0.5, seed=3 * k + n, a="int", b="int", c="int", lda=lda)
    assert _plan(p)["a_in_kernel"] == int(a_split)
    _run(p, exact=True)


def test_unaligned_lda_falls_back_to_pre_pass(monkeypatch):
    """TMA needs 16-byte rows: with lda % 4 != 0 A is split by the pre-pass
    even when the in-kernel split is requested."""
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", "1")
    p = inputs.make_problem(300, 200, 777, alpha=1.0, beta=0.0, seed=5, a="normal", b="normal")
    assert p.lda == 777 and _plan(p)["a_in_kernel"] == 0
    _run(p)


def test_in_kernel_split_is_deterministic(monkeypatch):
    """Repeated calls give identical bits (the split and the MMA order are
    fixed); the in-kernel and pre-pass splits differ only in how hi is
    rounded, both within the bound."""
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", "1")
    p = inputs.make_problem(700, 384, 1500, alpha=1.0, beta=0.0, seed=11, a="normal", b="normal", lda=1500)
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    outs = []
    for _ in range(3):
        C = torch.zeros(p.m, p.n, device="cuda")
        binding.sgemm_ex(A, B, C, 1.0, 0.0, path=TC)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_tensor_core_reads_fp32_operands_truncated_to_tf32():
    """The in-kernel split relies on a kind::tf32 MMA reading an FP32
    operand with its low 13 mantissa bits dropped: C = X * I through the
    split-GEMM call (X as the hi operand, every lo zero) must equal X
    truncated to TF32, including values on the rounding boundaries."""
    import numpy as np
    m = n = k = 256
    rng = np.random.default_rng(1)
    X = rng.standard_normal((m, k)).astype(np.float32)
    bits = X.view(np.uint32)
    bits[:, :6] = (bits[:, :6] & ~np.uint32(0x1FFF)) | np.array([0x1000, 0x0FFF, 0x1001, 0x1FFF, 1, 0], np.uint32)
    ka = binding.ka_of(k)
    x_hi = torch.from_numpy(X.copy()).cuda().reshape(-1)
    zeros_a = torch.zeros(m * ka, device="cuda")
    eye = torch.eye(n, ka, device="cuda").reshape(-1)
    zeros_b = torch.zeros(n * ka, device="cuda")
    C = torch.zeros(m, n, device="cuda")
    st = binding.tf32x3_split_gemm_raw(m, n, k, 1.0, x_hi.data_ptr(), zeros_a.data_ptr(), eye.data_ptr(),
                                       zeros_b.data_ptr(), 0.0, C.data_ptr(), n,
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    truncated = (X.view(np.uint32) & ~np.uint32(0x1FFF)).view(np.float32)
    assert np.array_equal(C.cpu().numpy(), truncated)
