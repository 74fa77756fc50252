"""GPU parity of stream-K scheduling (one CTA per SM, each an equal share of
the slab sequence of all tiles; a tile shared by several CTAs is finished
by the last of them from their partial sums in a workspace), pinned with
the library's tuning variable SGEMM_GB300_STREAM_K, against the FP64
oracle: 256-wide, 128-wide and transposed tiles, A split in the kernel and
by the pre-pass, ragged shapes, beta != 0, tiles shared by 2-3 CTAs and by
dozens, integer twins bit-exact, and repeatability; and the form that cuts
each tile left after the full waves into S equal k parts (one per CTA,
SGEMM_GB300_SK_PARTS) on the same kinds of tiles."""
import pytest
import torch

from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import Placed, check_full

pytestmark = pytest.mark.gpu

TC = binding.PATH_TF32X3


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(autouse=True)
def _clean_env(monkeypatch):
    for v in ("SGEMM_GB300_STREAM_K", "SGEMM_GB300_TRANS", "SGEMM_GB300_TILE_N", "SGEMM_GB300_SPLIT_A_IN",
              "SGEMM_GB300_SPLIT_K", "SGEMM_GB300_SK_PARTS"):
        monkeypatch.delenv(v, raising=False)


def _plan(p):
    st, plan = binding.plan(p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, path=TC,
                            num_sms=0)
    assert st == 0
    return plan


def _run(p, exact=False):
    pl = Placed(p)
    st = pl.run(TC)
    assert st == 0, binding.status_string(st)
    C, guard_ok = pl.result()
    assert guard_ok, "a write landed outside the m x n window of C"
    assert pl.inputs_untouched(), "A or B was modified"
    ok, worst, where = check_full(p, C, exact=exact)
    assert ok, f"worst |C - r| / tol = {worst} at {where}"
    return C


CASES = [
    # m, n, k, lda, beta, extra tuning variables
    (2048, 2048, 512, None, 0.0, {}),                              # 128 tiles of 128 x 256
    (1000, 1500, 777, 780, 0.5, {}),                               # ragged, A split in the kernel
    (1000, 1500, 777, None, 0.5, {}),                              # lda = 777: A split by the pre-pass
    (3000, 128, 1000, None, -1.0, {"SGEMM_GB300_TRANS": "0"}),     # 128 x 128 tiles
    (4096, 100, 1000, None, 2.0, {"SGEMM_GB300_TRANS": "1"}),      # transposed 256 x 128 tiles
    (2048, 2048, 64, None, 0.0, {}),                               # 4 slabs per tile: up to 3 CTAs per tile
    (256, 256, 8192, None, 0.5, {}),                               # 2 tiles shared by ~76 CTAs each
]


@pytest.mark.parametrize("sk", ["1", "0"], ids=["stream_k", "tiles"])
@pytest.mark.parametrize("m,n,k,lda,beta,env", CASES)
def test_stream_k_matches_oracle(monkeypatch, sk, m, n, k, lda, beta, env):
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", sk)
    for key, val in env.items():
        monkeypatch.setenv(key, val)
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=beta, seed=m + 7 * n + k, a="normal", b="uniform",
                            c="uniform" if beta else None, lda=lda)
    plan = _plan(p)
    assert (plan["stream_k"] > 0) == (sk == "1"), plan
    _run(p)


@pytest.mark.parametrize("m,n,k", [(2048, 2048, 512), (1000, 1500, 777), (256, 256, 8192)])
def test_stream_k_integer_twin_bit_exact(monkeypatch, m, n, k):
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "1")
    p = inputs.make_problem(m, n, k, alpha=2.0, beta=0.5, seed=3 * m + k, a="int", b="int", c="int",
                            lda=(k + 3) // 4 * 4)
    assert _plan(p)["stream_k"] > 0
    _run(p, exact=True)


def test_stream_k_is_deterministic(monkeypatch):
    """The last CTA of a shared tile adds the partials in k order, so the
    result does not depend on which CTA finishes last."""
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "1")
    p = inputs.make_problem(1000, 1500, 777, alpha=1.0, beta=0.0, seed=17, a="normal", b="normal", lda=780)
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    outs = []
    for _ in range(4):
        C = torch.zeros(p.m, p.n, device="cuda")
        binding.sgemm_ex(A[:, :p.k], B, C, 1.0, 0.0, path=TC)
        outs.append(C)
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


PARTS_CASES = [
    # m, n, k, lda, beta, extra tuning variables, S expected on 152 SMs
    (2432, 4608, 256, None, 0.0, {}, 4),                            # 342 tiles of 128 x 256 = 2 x 152 + 38
    (2400, 4600, 250, None, 0.5, {}, 4),                            # the same tiles, ragged in m, n and k
    (2432, 4608, 256, 257, 0.5, {}, 4),                             # lda odd: A read in row phases
    (25600, 128, 64, None, -1.0, {"SGEMM_GB300_TRANS": "0"}, 3),    # 200 tiles of 128 x 128 = 152 + 48
    (51200, 100, 64, None, 2.0, {"SGEMM_GB300_TRANS": "1"}, 3),     # 200 transposed 256 x 128 tiles
    (16384, 128, 2048, None, 1.0, {}, 2),                           # no full wave: 64 tiles, 2 parts each
]


@pytest.mark.parametrize("m,n,k,lda,beta,env,S", PARTS_CASES)
def test_stream_k_parts_match_oracle(monkeypatch, m, n, k, lda, beta, env, S):
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "1")
    monkeypatch.setenv("SGEMM_GB300_SK_PARTS", "1")
    for key, val in env.items():
        monkeypatch.setenv(key, val)
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=beta, seed=m + 3 * n + k, a="normal", b="uniform",
                            c="uniform" if beta else None, lda=lda)
    plan = _plan(p)
    assert plan["stream_k"] > 0, plan
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert plan["sk_parts"] == S, plan
    assert plan["sk_parts"] >= 2, plan
    _run(p)


def test_stream_k_parts_integer_twin_bit_exact_and_repeatable(monkeypatch):
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "1")
    monkeypatch.setenv("SGEMM_GB300_SK_PARTS", "1")
    p = inputs.make_problem(2432, 4608, 256, alpha=2.0, beta=0.5, seed=29, a="int", b="int", c="int")
    assert _plan(p)["sk_parts"] >= 2
    C = _run(p, exact=True)
    C2 = _run(p, exact=True)
    assert torch.equal(torch.as_tensor(C), torch.as_tensor(C2))
