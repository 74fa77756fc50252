"""When a call runs a split pass (an operand TMA cannot read as stored, or
the split pass forced), the tensor-core GEMM is launched as a programmatic
dependent of it (its set-up overlaps the split's tail; its TMA producer
waits for the split before reading the split operands).  That gives the
same bits as a normal launch, and matches the oracle, for one-wave GEMMs
where the library uses it: whole tiles, split-K clusters, transposed
tiles, either operand split first, beta != 0."""
import pytest
import torch

from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import Placed, check_full

pytestmark = pytest.mark.gpu

TC = binding.PATH_TF32X3


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("m,n,k,lda,beta,env", [
    (2048, 2048, 512, None, 0.0, {"SGEMM_GB300_SPLIT_B_IN": "0"}),   # 128 whole tiles, B split first
    (1000, 1500, 777, None, 0.5, {"SGEMM_GB300_SPLIT_A_IN": "0"}),   # lda = 777, A split first: split-K cluster
    (3000, 100, 2048, None, 1.0, {"SGEMM_GB300_SPLIT_B_IN": "0"}),   # transposed tiles
    (512, 512, 512, None, -2.0, {"SGEMM_GB300_SPLIT_A_IN": "0", "SGEMM_GB300_SPLIT_B_IN": "0"}),
])
def test_dependent_launch_matches_normal_launch(monkeypatch, m, n, k, lda, beta, env):
    for key, val in env.items():
        monkeypatch.setenv(key, val)
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=beta, seed=m + n + 3 * k, a="normal", b="uniform",
                            c="uniform" if beta else None, lda=lda)
    st, plan = binding.plan(p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, path=TC,
                            num_sms=0)
    # a split pass runs, and the GEMM fits in one wave
    assert st == 0 and not (plan["a_in_kernel"] and plan["b_in_kernel"]) and plan["grid"] <= 152
    outs = []
    for pdl in ("1", "0"):
        monkeypatch.setenv("SGEMM_GB300_PDL", pdl)
        pl = Placed(p)
        st = pl.run(TC)
        assert st == 0, binding.status_string(st)
        C, guard_ok = pl.result()
        assert guard_ok and pl.inputs_untouched()
        outs.append(C)
    ok, worst, where = check_full(p, outs[0])
    assert ok, f"worst |C - r| / tol = {worst} at {where}"
    assert (outs[0] == outs[1]).all()
