"""GPU parity of sgemm_strided_batched: every problem of a strided batch
against the FP64 oracle, on both paths, including shared (stride 0)
operands, transposed operands, gaps between C matrices, split-K inside a
batch and batches of many small problems."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import SENTINEL

pytestmark = pytest.mark.gpu

PATHS = {"ffma": binding.PATH_FFMA, "tf32x3": binding.PATH_TF32X3}


def run_batch(batch, m, n, k, path, *, op_a=0, op_b=0, share_a=False, share_b=False, gap=(0, 0, 3),
              alpha=1.5, beta=0.5, dist="normal", seed=0, exact=False, check=None):
    rng_seed = seed
    probs = [inputs.make_problem(m, n, k, alpha=alpha, beta=beta, seed=rng_seed + b, a=dist,
                                 b="int" if dist == "int" else "uniform", c="int" if dist == "int" else "uniform")
             for b in range(batch)]
    if share_a:
        for p in probs:
            p.A = probs[0].A
    if share_b:
        for p in probs:
            p.B = probs[0].B
    a_st = [p.A[:, :k] if op_a == 0 else np.ascontiguousarray(p.A[:, :k].T) for p in probs]
    b_st = [p.B[:, :n] if op_b == 0 else np.ascontiguousarray(p.B[:, :n].T) for p in probs]
    lda, ldb, ldc = a_st[0].shape[1], b_st[0].shape[1], n
    sa = 0 if share_a else a_st[0].size + gap[0]
    sb = 0 if share_b else b_st[0].size + gap[1]
    sc = m * ldc + gap[2]

    def pack(mats, stride):
        size = stride * (len(mats) - 1) + mats[0].size if stride else mats[0].size
        buf = np.full(size + 64, SENTINEL, np.float32)
        for b, x in enumerate(mats if stride else mats[:1]):
            buf[b * stride: b * stride + x.size] = x.reshape(-1)
        return buf

    A = torch.from_numpy(pack(a_st, sa)).cuda()
    B = torch.from_numpy(pack(b_st, sb)).cuda()
    Ch = pack([p.C0[:, :n] for p in probs], sc)
    C = torch.from_numpy(Ch.copy()).cuda()
    st = binding.sgemm_strided_batched_raw(op_a, op_b, m, n, k, alpha, A.data_ptr(), lda, sa, B.data_ptr(), ldb, sb,
                                           beta, C.data_ptr(), ldc, sc, batch,
                                           torch.cuda.current_stream().cuda_stream, path)
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    out = C.cpu().numpy()
    # the gaps between C matrices and the tail are untouched
    mask = np.ones(out.size, bool)
    for b in range(batch):
        mask[b * sc: b * sc + m * ldc] = False
    assert np.array_equal(out[mask], Ch[mask]), "a write landed between the batch's C matrices"
    for b in (range(batch) if check is None else check):
        p = probs[b]
        got = out[b * sc: b * sc + m * ldc].reshape(m, ldc)[:, :n]
        R, E, Rf = oracle.sgemm_f64(m, n, k, alpha, p.A[:, :k], k, p.B[:, :n], n, beta, p.C0[:, :n], n)
        if exact:
            assert np.array_equal(got, Rf), f"problem {b}"
        else:
            ok, worst, where = oracle.within_tolerance(got, R, E, beta, p.C0[:, :n])
            assert ok, f"problem {b}: worst {worst} at {where}"


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
@pytest.mark.parametrize("batch,m,n,k", [(5, 130, 257, 77), (3, 256, 256, 256), (7, 33, 65, 129), (2, 1000, 1500, 777)])
def test_strided_batch(batch, m, n, k, path):
    run_batch(batch, m, n, k, path, seed=batch * 1000 + m)


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
@pytest.mark.parametrize("share", ["a", "b"])
def test_shared_operand(share, path):
    run_batch(4, 200, 150, 96, path, share_a=share == "a", share_b=share == "b", seed=17)


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
@pytest.mark.parametrize("op_a,op_b", [(1, 0), (0, 1), (1, 1)], ids=["TN", "NT", "TT"])
def test_transposed_batch(op_a, op_b, path):
    run_batch(3, 150, 170, 90, path, op_a=op_a, op_b=op_b, seed=23)


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
def test_batch_integer_twin_bit_exact(path):
    run_batch(4, 129, 200, 300, path, alpha=2.0, beta=0.5, dist="int", seed=31, exact=True)


def test_split_k_inside_a_batch():
    """A batch whose tiles are few enough that each problem's tile is split
    over a cluster."""
    st, plan = binding.plan(256, 256, 8192, lda=8192, path=binding.PATH_TF32X3, num_sms=0)
    assert plan["split_k"] > 1
    run_batch(2, 256, 256, 8192, binding.PATH_TF32X3, seed=41)


@pytest.mark.parametrize("k,share_a,gap_a", [(77, True, 0), (96, False, 1), (77, False, 2)],
                         ids=["lda77_shared", "stride_misaligned", "lda77_gap"])
def test_phased_a_inside_a_batch(k, share_a, gap_a):
    """An A that TMA cannot read -- rows 77 floats apart, or 16-byte rows
    whose problems are 1 float further apart than a multiple of 4 -- is
    read by the GEMM in row phases from problem blockIdx.y's matrix (or the
    one shared matrix)."""
    m, n = 200, 150
    st, plan = binding.plan(m, n, k, lda=k, path=binding.PATH_TF32X3, num_sms=0)
    assert st == 0 and plan["a_in_kernel"] == 1 and plan["trans"] == 0
    run_batch(3, m, n, k, binding.PATH_TF32X3, share_a=share_a, gap=(gap_a, 0, 3), seed=61 + k)


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
def test_many_small_problems(path):
    run_batch(300, 48, 40, 24, path, seed=53, check=[0, 1, 150, 298, 299])


@pytest.mark.parametrize("path", PATHS.values(), ids=PATHS.keys())
def test_bmm_binding_with_views(path):
    torch.manual_seed(5)
    A = torch.randn(6, 70, 50, device="cuda")
    Bt = torch.randn(6, 90, 50, device="cuda")      # B = Bt^T per problem: 50 x 90
    C = torch.zeros(6, 70, 90, device="cuda")
    binding.bmm(A, Bt.transpose(1, 2), C, path=path)
    ref = A.double() @ Bt.transpose(1, 2).double()
    E = A.double().abs() @ Bt.transpose(1, 2).double().abs()
    assert torch.all((C.double() - ref).abs() <= 1e-5 * E)


def test_zero_batch_is_a_noop():
    assert binding.sgemm_strided_batched_raw(0, 0, 4, 4, 4, 1.0, 0, 4, 0, 0, 4, 0, 0.0, 0, 4, 16, 0) == 0
