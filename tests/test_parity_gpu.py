"""GPU parity: the CUDA path through the C ABI against the FP64 oracle on the
same seeded inputs.

* real-valued inputs: |C - r| <= 1e-5 * sum_t |A_it||B_tj| + 1e-6 * |beta C0|
  on every element (sizes the oracle finishes in seconds) or on 4096 sampled
  outputs plus every partial-tile edge (the 8192^3 and 16384x128x8192
  workloads);
* integer twins (entries in {-4..4}): bit-exact, every product and partial
  sum being an integer below 2^24;
* guard bands around C and the row gaps of padded leading dimensions must
  survive, and A and B must not be written.
"""
import numpy as np
import pytest
import torch

from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import Placed, check_full, check_sampled

pytestmark = pytest.mark.gpu

PATHS = [binding.PATH_FFMA, binding.PATH_TF32X3]
PATH_IDS = {binding.PATH_FFMA: "ffma", binding.PATH_TF32X3: "tf32x3", binding.PATH_AUTO: "auto"}


def path_runs(path, p, offs=(0, 0, 0)):
    st, _ = binding.plan(p.m, p.n, p.k, p.alpha, 16 + 4 * offs[0], p.lda, 16 + 4 * offs[1], p.ldb, p.beta,
                         16 + 4 * offs[2], p.ldc, path=path)
    return st != 99


def run_and_check(p, path, offs=(0, 0, 0), exact=False, sample=None):
    if not path_runs(path, p, offs):
        pytest.skip(f"path {PATH_IDS[path]} does not take this problem")
    pl = Placed(p, offs)
    st = pl.run(path)
    assert st == 0, binding.status_string(st)
    C, guard_ok = pl.result()
    assert guard_ok, "a write landed outside the m x n window of C"
    assert pl.inputs_untouched(), "A or B was modified"
    if sample is None:
        ok, worst, where = check_full(p, C, exact=exact)
    else:
        rows, cols = sample
        ok, worst, where = check_sampled(p, C, rows, cols, exact=exact)
    assert ok, f"worst |C - r| / tol = {worst} at {where}"
    return C


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


# ---------------------------------------------------------------- the five workloads

SMALL = ["256^3", "2048^3", "1000x1500x777"]
LARGE = ["8192^3", "16384x128x8192"]


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("name", SMALL)
def test_workload_full(name, path):
    run_and_check(inputs.workload(name), path)


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("name", SMALL)
def test_workload_integer_twin_bit_exact(name, path):
    run_and_check(inputs.workload(name, twin=True), path, exact=True)


@pytest.mark.parametrize("path", PATHS + [binding.PATH_AUTO], ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("name", LARGE)
def test_workload_sampled(name, path):
    p = inputs.workload(name)
    run_and_check(p, path, sample=inputs.sample_indices(p.m, p.n, 4096, seed=p.seed + 1000))


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("name", LARGE)
def test_workload_integer_twin_sampled_bit_exact(name, path):
    p = inputs.workload(name, twin=True)
    run_and_check(p, path, exact=True, sample=inputs.sample_indices(p.m, p.n, 4096, seed=p.seed + 1000))


@pytest.mark.parametrize("path", PATHS + [binding.PATH_AUTO], ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("name", LARGE)
def test_workload_every_output_by_projection(name, path):
    """Every output of the full-size workloads, through random projections
    (Freivalds' check, in FP64 on the GPU): C x against alpha A (B x) +
    beta C0 x and y^T C against alpha (y^T A) B + beta y^T C0, each row
    (column) within the sum over it of the per-element FP32 bound,
    1e-5 |alpha| (|A| (|B| |x|)) + 1e-6 |beta| (|C0| |x|).  A tile written
    wrong, twice or not at all moves its 128 rows (columns) far outside it;
    with beta = 0, C starts as the sentinel and none may be left."""
    import gpu_util
    p = inputs.workload(name)
    if not path_runs(path, p):
        pytest.skip(f"path {PATH_IDS[path]} does not take this problem")
    A = torch.from_numpy(np.ascontiguousarray(p.A[:, :p.k])).cuda()
    B = torch.from_numpy(np.ascontiguousarray(p.B[:, :p.n])).cuda()
    C0 = torch.from_numpy(np.ascontiguousarray(p.C0[:, :p.n])).cuda()
    C = C0.clone() if p.beta != 0 else torch.full((p.m, p.n), float(gpu_util.SENTINEL), device="cuda")
    binding.sgemm_ex(A, B, C, p.alpha, p.beta, path=path)
    torch.cuda.synchronize()
    if p.beta == 0:
        assert not bool((C == float(gpu_util.SENTINEL)).any()), "an output was never written"
    rx, ry = gpu_util.projection_ratios(A, B, C0, C, p.alpha, p.beta, p.seed + 77)
    assert rx <= 1.0 and ry <= 1.0, f"projection residual / bound: rows {rx}, columns {ry}"


# ---------------------------------------------------------------- edges and tails

EDGE = [1, 3, 4, 5, 31, 127, 128, 129, 200]


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("m,n,k", [
    (1, 1, 1), (1, 129, 5), (129, 1, 3), (3, 5, 4), (127, 128, 129), (128, 128, 128),
    (129, 129, 129), (200, 31, 1), (5, 200, 300), (255, 257, 33), (64, 384, 16), (385, 130, 47),
])
def test_ragged_shapes(m, n, k, path):
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=-0.75, seed=m * 7 + n * 11 + k, c="uniform")
    run_and_check(p, path)


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
def test_ragged_integer_sweep_bit_exact(path):
    rng = np.random.default_rng(2024)
    for trial in range(12):
        m, n, k = (int(rng.choice(EDGE)) for _ in range(3))
        p = inputs.make_problem(m, n, k, alpha=2.0, beta=0.5, seed=500 + trial, a="int", b="int", c="int")
        run_and_check(p, path, exact=True)


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
def test_padded_leading_dimensions(path):
    p = inputs.make_problem(300, 200, 150, alpha=1.0, beta=1.0, seed=9, c="uniform",
                            lda=161, ldb=203, ldc=260)
    run_and_check(p, path)


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1)])
def test_misaligned_pointers(offs, path):
    p = inputs.make_problem(260, 140, 90, alpha=0.5, beta=2.0, seed=10, c="normal")
    run_and_check(p, path, offs=offs)


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
def test_unaligned_lda_workload_twin(path):
    """lda = 777 (rows 3108 bytes apart, not a multiple of 16) with ragged
    m, n: the 1000 x 1500 x 777 workload's layout on integer inputs."""
    p = inputs.workload("1000x1500x777", twin=True)
    assert p.lda == 777
    run_and_check(p, path, exact=True)


@pytest.mark.parametrize("path,m,n,k", [
    (binding.PATH_FFMA, 384, 200, 8192), (binding.PATH_FFMA, 130, 520, 8192),
    (binding.PATH_TF32X3, 384, 200, 8192), (binding.PATH_TF32X3, 256, 256, 32768),
    (binding.PATH_TF32X3, 130, 520, 65536), (binding.PATH_AUTO, 256, 256, 32768),
], ids=lambda v: PATH_IDS.get(v, str(v)) if isinstance(v, int) and v < 3 else str(v))
def test_nonnegative_long_k(path, m, n, k):
    """Non-negative operands: every partial sum grows with t, so an
    accumulation whose rounding is biased (not round-to-nearest) drifts
    linearly in k and shows here first.  The FFMA path sums each output
    sequentially in FP32 and is held to the bound up to k = 8192 (the
    largest workload); the tensor-core path, which accumulates 128-deep
    chunks in TMEM and adds the chunks in FP32 registers, to k = 65536."""
    p = inputs.make_problem(m, n, k, alpha=1.0, beta=0.0, seed=k + m, a="uniform01", b="uniform01")
    run_and_check(p, path)


# ---------------------------------------------------------------- alpha, beta, k = 0

@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
def test_beta_zero_ignores_nan_c(path):
    p = inputs.make_problem(150, 170, 60, alpha=1.0, beta=0.0, seed=11, c=None, c_fill=float("nan"))
    C = run_and_check(p, path)
    assert np.all(np.isfinite(C))


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
def test_alpha_zero_scales_c_only(path):
    p = inputs.make_problem(70, 90, 33, alpha=0.0, beta=-1.5, seed=12, c="uniform")
    p.A[:] = np.nan
    p.B[:] = np.nan
    C = run_and_check(p, path)
    np.testing.assert_array_equal(C, (np.float32(-1.5) * p.C0[:, :p.n]).astype(np.float32))


@pytest.mark.parametrize("path", PATHS, ids=lambda p: PATH_IDS[p])
def test_k_zero(path):
    for beta in (0.0, 3.0):
        p = inputs.make_problem(33, 65, 0, alpha=1.0, beta=beta, seed=13, c="uniform")
        C = run_and_check(p, path)
        np.testing.assert_array_equal(C, (np.float32(beta) * p.C0[:, :p.n]).astype(np.float32))


def test_empty_output_launches_nothing():
    for m, n in ((0, 5), (5, 0), (0, 0)):
        assert binding.sgemm_raw(m, n, 7, 1.0, 0, 7, 0, max(n, 1), 0.0, 0, max(n, 1)) == 0


# ---------------------------------------------------------------- torch-facing binding

def test_binding_on_tensor_views():
    torch.manual_seed(0)
    big = torch.randn(300, 400, device="cuda")
    A = big[10:110, 5:77]           # 100 x 72, row stride 400
    B = torch.randn(72, 90, device="cuda")
    C = torch.zeros(100, 128, device="cuda")[:, :90]
    binding.sgemm(A, B, C)
    ref = (A.double() @ B.double()).float()
    E = (A.double().abs() @ B.double().abs())
    assert torch.all((C.double() - ref.double()).abs() <= 1e-5 * E + 1e-30)


def test_stream_ordering():
    """Work enqueued on a side stream is ordered by that stream."""
    s = torch.cuda.Stream()
    p = inputs.workload("256^3", twin=True)
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C = torch.full((256, 256), float("nan"), device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.sgemm(A, B, C)
        out = C.clone()
    torch.cuda.synchronize()
    want = (A.double() @ B.double()).float()
    assert torch.equal(out, want)


# ---------------------------------------------------------------- 3xTF32 split operands

def test_tf32x3_split_operands(monkeypatch):
    """The split calls produce hi = TF32(x) (low 13 mantissa bits zero),
    lo = TF32(x - hi), with |x - hi - lo| <= 2^-22 |x| and |lo| <= 2^-11 |x|;
    B comes out transposed; the split GEMM equals the one-call path bit for
    bit when that path splits both operands with the split pass too (same
    kernels, same operands)."""
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", "0")
    monkeypatch.setenv("SGEMM_GB300_SPLIT_B_IN", "0")
    p = inputs.make_problem(300, 260, 150, alpha=1.25, beta=0.5, seed=31, a="normal", b="uniform", c="uniform")
    ka = binding.ka_of(p.k)
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    a_hi = torch.zeros(p.m * ka, device="cuda")
    a_lo = torch.zeros_like(a_hi)
    b_hi = torch.zeros(p.n * ka, device="cuda")
    b_lo = torch.zeros_like(b_hi)
    binding.tf32x3_split_a(A, a_hi, a_lo)
    binding.tf32x3_split_b(B, b_hi, b_lo)
    torch.cuda.synchronize()
    ah = a_hi.view(p.m, ka)[:, :p.k].cpu().numpy()
    al = a_lo.view(p.m, ka)[:, :p.k].cpu().numpy()
    bh = b_hi.view(p.n, ka)[:, :p.k].cpu().numpy()
    bl = b_lo.view(p.n, ka)[:, :p.k].cpu().numpy()
    for x, hi, lo in ((p.A.astype(np.float64), ah, al), (p.B.T.astype(np.float64), bh, bl)):
        assert np.all(hi.view(np.uint32) & 0x1FFF == 0) and np.all(lo.view(np.uint32) & 0x1FFF == 0)
        assert np.all(np.abs(x - hi) <= 2.0 ** -11 * np.abs(x))
        assert np.all(np.abs(x - hi.astype(np.float64) - lo.astype(np.float64)) <= 2.0 ** -22 * np.abs(x))
    C1 = torch.from_numpy(p.C0).cuda()
    C2 = C1.clone()
    st = binding.tf32x3_split_gemm_raw(p.m, p.n, p.k, p.alpha, a_hi.data_ptr(), a_lo.data_ptr(), b_hi.data_ptr(),
                                       b_lo.data_ptr(), p.beta, C1.data_ptr(), p.ldc,
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0
    binding.sgemm_ex(A, B, C2, p.alpha, p.beta, path=binding.PATH_TF32X3)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


def test_device_status_clear_after_runs():
    """No bounded wait gave up during the tests above."""
    import ctypes
    from dense_fp32_gemm_06_gb300 import _native
    flag = ctypes.c_int(-1)
    assert _native.load().sgemm_device_status(ctypes.byref(flag), 0) == 0
    assert flag.value == 0


# ---------------------------------------------------------------- split-K clusters

@pytest.mark.parametrize("m,n,k,beta", [
    (256, 256, 8192, 0.0), (300, 700, 5000, 0.75), (129, 257, 4096, -1.0), (1000, 1500, 777, 0.5),
    (64, 64, 65536, 0.0), (400, 300, 3000, 2.0),
])
def test_split_k_clusters(monkeypatch, m, n, k, beta):
    """Problems with few tiles split k over a cluster of CTAs that reduce
    their partial tiles through distributed shared memory (stream-K, which
    the plan may prefer for some of these shapes, is pinned off)."""
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "0")
    st, plan = binding.plan(m, n, k, lda=k, path=binding.PATH_TF32X3, num_sms=0)
    if plan["split_k"] == 1:   # this device's cluster capacity favours whole tiles here: split anyway
        monkeypatch.setenv("SGEMM_GB300_SPLIT_K", "3")
        st, plan = binding.plan(m, n, k, lda=k, path=binding.PATH_TF32X3, num_sms=0)
    assert st == 0 and plan["split_k"] > 1, plan
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=beta, seed=m + n + k, a="normal", b="uniform",
                            c="uniform" if beta else None)
    run_and_check(p, binding.PATH_TF32X3)


@pytest.mark.parametrize("m,n,k", [(256, 256, 8192), (300, 700, 5000), (1000, 1500, 777)])
def test_split_k_integer_twin_bit_exact(monkeypatch, m, n, k):
    """Partial sums of integers are exact, so the split result is too."""
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "0")
    st, plan = binding.plan(m, n, k, lda=k, path=binding.PATH_TF32X3, num_sms=0)
    if plan["split_k"] == 1:   # as above
        monkeypatch.setenv("SGEMM_GB300_SPLIT_K", "3")
        st, plan = binding.plan(m, n, k, lda=k, path=binding.PATH_TF32X3, num_sms=0)
    assert st == 0 and plan["split_k"] > 1
    p = inputs.make_problem(m, n, k, alpha=2.0, beta=0.5, seed=7 * k, a="int", b="int", c="int")
    run_and_check(p, binding.PATH_TF32X3, exact=True)


def test_split_k_is_deterministic():
    """The cluster reduction adds partials in a fixed order: repeated calls
    give identical bits."""
    p = inputs.make_problem(300, 700, 5000, alpha=1.0, beta=0.0, seed=99, a="normal", b="normal")
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    outs = []
    for _ in range(3):
        C = torch.zeros(p.m, p.n, device="cuda")
        binding.sgemm_ex(A, B, C, 1.0, 0.0, path=binding.PATH_TF32X3)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
