"""GPU parity of the tensor-core path with each operand split inside the
GEMM kernel (the raw FP32 operand loaded by TMA as stored -- A K-major, B
MN-major -- and read as its own hi part, lo computed in shared memory) or
by the separate split pass, pinned through the library's tuning variables
SGEMM_GB300_SPLIT_A_IN / SGEMM_GB300_SPLIT_B_IN and checked against the FP64
oracle: ragged tiles, k tails that are not a multiple of the 16-deep slab,
split-K clusters, beta != 0, padded leading dimensions, and bit-exact
integer twins.  Also the property the in-kernel split rests on: the tensor
core reads an FP32 operand, K-major or MN-major, with its low 13 mantissa
bits dropped."""
import numpy as np
import pytest
import torch

from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import Placed, check_full

pytestmark = pytest.mark.gpu

TC = binding.PATH_TF32X3


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(params=[("1", "1"), ("1", "0"), ("0", "1"), ("0", "0")],
                ids=["both_in_kernel", "a_in_kernel", "b_in_kernel", "pre_pass"])
def split(request, monkeypatch):
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", request.param[0])
    monkeypatch.setenv("SGEMM_GB300_SPLIT_B_IN", request.param[1])
    return request.param[0] == "1", request.param[1] == "1"


def _expect_plan(p, split):
    """The requested in-kernel splits, where TMA can read the operand (its
    rows 16-byte aligned; the guarded buffers start 16-byte aligned)."""
    plan = _plan(p)
    assert plan["a_in_kernel"] == int(split[0] and p.lda % 4 == 0), plan
    assert plan["b_in_kernel"] == int(split[1] and p.ldb % 4 == 0), plan
    assert plan["threads"] == 384, plan


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
def test_in_kernel_and_pre_pass_split_match_oracle(split, m, n, k, lda, beta):
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=beta, seed=m * 7 + n + k, a="normal", b="uniform",
                            c="uniform" if beta else None, lda=lda)
    _expect_plan(p, split)
    _run(p)


@pytest.mark.parametrize("m,n,k", [(1000, 300, 777), (129, 257, 4096), (512, 512, 2048)])
def test_in_kernel_split_integer_twin_bit_exact(split, m, n, k):
    """hi(x) = x and lo(x) = 0 for small integers, so every product and
    partial sum is exact whichever side splits A and B."""
    lda = (k + 3) // 4 * 4
    ldb = (n + 3) // 4 * 4
    p = inputs.make_problem(m, n, k, alpha=2.0, beta=0.5, seed=3 * k + n, a="int", b="int", c="int", lda=lda,
                            ldb=ldb)
    _expect_plan(p, split)
    _run(p, exact=True)


def test_unaligned_rows(monkeypatch):
    """TMA needs 16-byte rows: with ldb % 4 != 0 B is split by the split
    pass even when the in-kernel split is requested, while A is still read
    as stored; with lda % 4 != 0 TMA reads A in four row phases (rows j,
    j + 4, ...: 16-byte row pitch) and the splitter warps shift each row
    into place and split it."""
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", "1")
    monkeypatch.setenv("SGEMM_GB300_SPLIT_B_IN", "1")
    p = inputs.make_problem(300, 200, 777, alpha=1.0, beta=0.0, seed=5, a="normal", b="normal")
    assert p.lda == 777 and (_plan(p)["a_in_kernel"], _plan(p)["b_in_kernel"]) == (1, 1)
    _run(p)
    p = inputs.make_problem(300, 203, 776, alpha=1.0, beta=0.0, seed=6, a="normal", b="normal")
    assert p.ldb == 203 and (_plan(p)["a_in_kernel"], _plan(p)["b_in_kernel"]) == (1, 0)
    _run(p)


# A whose rows TMA cannot read as one tensor, read in row phases and put
# into the swizzled stage slots by the splitter warps: the plan each case
# runs in a comment
@pytest.mark.parametrize("m,n,k,lda,off_a,beta", [
    (1000, 1500, 777, 777, 0, 0.5),      # the 1000 x 1500 x 777 workload's layout: split-K 3
    (300, 200, 777, 777, 1, 0.0),        # base 4 bytes past 16-byte alignment too
    (129, 257, 4096, 4097, 2, -1.0),     # split-K 8, B split first (ldb = 257)
    (2048, 2048, 2048, 2049, 0, 0.0),    # 128 wide tiles, B split first (above 2^31)
    (3000, 2000, 999, 999, 3, 1.0),      # stream-K over 152 CTAs
    (128, 128, 5, 5, 0, 0.0),            # one slab, k = 5
    (200, 300, 1, 1, 1, 0.5),            # k = 1
    (640, 1024, 2047, 2047, 0, 2.0),     # split-K 6, k % 16 = 15
    (1000, 300, 780, 780, 1, 0.0),       # 16-byte rows, base misaligned
])
def test_phased_a_matches_oracle(monkeypatch, m, n, k, lda, off_a, beta):
    for v in ("SGEMM_GB300_SPLIT_A_IN", "SGEMM_GB300_SPLIT_B_IN"):
        monkeypatch.delenv(v, raising=False)
    p = inputs.make_problem(m, n, k, alpha=0.75, beta=beta, seed=m + n + 3 * k, a="normal", b="uniform",
                            c="uniform" if beta else None, lda=lda)
    st, plan = binding.plan(p.m, p.n, p.k, p.alpha, 256 + 4 * off_a, p.lda, 256, p.ldb, p.beta, 256, p.ldc,
                            path=TC, num_sms=0)
    assert st == 0 and plan["a_in_kernel"] == 1 and plan["trans"] == 0 and plan["pair"] == 0, plan
    pl = Placed(p, off=(off_a, 0, 0))
    st = pl.run(TC)
    assert st == 0, binding.status_string(st)
    C, guard_ok = pl.result()
    assert guard_ok, "a write landed outside the m x n window of C"
    assert pl.inputs_untouched(), "A or B was modified"
    ok, worst, where = check_full(p, C)
    assert ok, f"worst |C - r| / tol = {worst} at {where}"
    assert binding.device_status() == 0


@pytest.mark.parametrize("m,n,k,lda", [(1000, 1500, 777, 777), (700, 512, 1001, 1003), (129, 130, 33, 33)])
def test_phased_a_integer_twin_bit_exact(monkeypatch, m, n, k, lda):
    """Integer operands through the phased A: exact products and sums, so
    any element put in the wrong place (a swizzle slip, a row, phase or
    shift error) changes the result."""
    for v in ("SGEMM_GB300_SPLIT_A_IN", "SGEMM_GB300_SPLIT_B_IN"):
        monkeypatch.delenv(v, raising=False)
    p = inputs.make_problem(m, n, k, alpha=2.0, beta=0.5, seed=k + 5 * n, a="int", b="int", c="int", lda=lda)
    assert _plan(p)["a_in_kernel"] == 1
    _run(p, exact=True)


def test_phased_a_identity_names_every_element(monkeypatch):
    """C = X * I with X[i][t] = i + 1024 t: every output is one element of A
    exactly, so an element put in the wrong row, k position or swizzle
    chunk shows as the wrong value (X has 1001 columns, lda = 1001)."""
    for v in ("SGEMM_GB300_SPLIT_A_IN", "SGEMM_GB300_SPLIT_B_IN"):
        monkeypatch.delenv(v, raising=False)
    m, k, n = 300, 1001, 1001
    X = (np.arange(m)[:, None] + 1024.0 * np.arange(k)[None, :]).astype(np.float32)
    I = np.eye(k, n, dtype=np.float32)
    Ad, Bd = torch.from_numpy(X).cuda(), torch.from_numpy(I).cuda()
    st, plan = binding.plan(m, n, k, 1.0, Ad.data_ptr(), k, Bd.data_ptr(), n, 0.0, 256, n, path=TC)
    assert st == 0 and plan["a_in_kernel"] == 1
    C = torch.full((m, n), -1.0, device="cuda")
    st = binding.sgemm_raw(m, n, k, 1.0, Ad.data_ptr(), k, Bd.data_ptr(), n, 0.0, C.data_ptr(), n,
                           torch.cuda.current_stream().cuda_stream, TC)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    bad = np.argwhere(got != X)
    assert bad.size == 0, [(int(i), int(j), float(got[i, j]), float(X[i, j])) for i, j in bad[:8]]


def test_in_kernel_split_is_deterministic(monkeypatch):
    """Repeated calls give identical bits (the split and the MMA order are
    fixed); the in-kernel and pre-pass splits differ only in how hi is
    rounded, both within the bound."""
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", "1")
    monkeypatch.setenv("SGEMM_GB300_SPLIT_B_IN", "1")
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


def _hi_plus_lo(X):
    """What the GEMM makes of a raw operand value x: hi = x with its low 13
    mantissa bits dropped (how the MMA reads FP32), lo = x - hi rounded to
    TF32 to nearest, ties away from zero (exact in FP32 arithmetic), and
    their sum, exact in FP32 (hi has 11 significant bits, lo at most 11
    more, 11 or more binary places below)."""
    import numpy as np
    bits = X.view(np.uint32)
    hi = (bits & ~np.uint32(0x1FFF)).view(np.float32)
    r = (X - hi).astype(np.float32)
    rb = r.view(np.uint32)
    lo = ((rb + np.uint32(0x1000)) & ~np.uint32(0x1FFF)).view(np.float32)   # |r| < 2^-10 |x|: no overflow
    return (hi.astype(np.float64) + lo.astype(np.float64)).astype(np.float32)


def _boundary_values(rows, cols, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((rows, cols)).astype(np.float32)
    bits = X.view(np.uint32)
    pats = np.array([0x1000, 0x0FFF, 0x1001, 0x1FFF, 1, 0, 0x17FF, 0x0800], np.uint32)
    bits[:, :8] = (bits[:, :8] & ~np.uint32(0x1FFF)) | pats
    return X


@pytest.mark.parametrize("op_a,op_b", [(0, 0), (0, 1), (1, 0)], ids=["B_mn_major", "B_k_major", "A_mn_major"])
def test_raw_operands_read_as_truncated_hi_plus_lo(monkeypatch, op_a, op_b):
    """With the identity as the other operand, every output is a single
    product: C = X exactly as the GEMM splits a raw X, hi = trunc(x) plus
    lo = tf32(x - hi), for X read MN-major (B stored k x n, or A stored
    k x m) or K-major (B stored n x k); values on the rounding boundaries
    included.  A tensor core that rounded an MN-major FP32 operand instead
    of truncating it would miss by up to 2^-11 |x|."""
    import numpy as np
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", "1")
    monkeypatch.setenv("SGEMM_GB300_SPLIT_B_IN", "1")
    n = k = m = 256
    X = _boundary_values(256, 256, 7 + op_a + 2 * op_b)
    eye = np.eye(256, dtype=np.float32)
    if op_a == 0:
        # C = I * op(B): op(B) = X, stored as X (k x n) or as X^T (n x k)
        A, B, want = eye, (X if op_b == 0 else np.ascontiguousarray(X.T)), _hi_plus_lo(X)
    else:
        # C = op(A) * I with op(A) = X stored as X^T (k x m)
        A, B, want = np.ascontiguousarray(X.T), eye, _hi_plus_lo(X)
    st, plan = binding.plan(m, n, k, 1.0, 256, 256, 256, 256, 0.0, 256, 256, path=TC)
    assert st == 0 and plan["a_in_kernel"] == 1 and plan["b_in_kernel"] == 1
    Ad = torch.from_numpy(A).cuda()
    Bd = torch.from_numpy(B).cuda()
    C = torch.zeros(m, n, device="cuda")
    st = binding.sgemm_op_raw(op_a, op_b, m, n, k, 1.0, Ad.data_ptr(), 256, Bd.data_ptr(), 256, 0.0, C.data_ptr(),
                              n, torch.cuda.current_stream().cuda_stream, TC)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]
