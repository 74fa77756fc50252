"""GPU parity of persistent whole tiles: for whole-tile plans of more than
one wave the library runs one CTA per SM, CTA g taking tiles g, g + 152,
... (the next tile's first chunks overlap the previous tile's epilogue).
Ragged shapes, beta != 0, an A read in row phases, 128-wide and transposed
tiles, integer twins bit for bit, and the same bits as one CTA per tile
(SGEMM_GB300_PERSIST=0)."""
import pytest
import torch

from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import Placed, check_full

pytestmark = pytest.mark.gpu

TC = binding.PATH_TF32X3


@pytest.fixture(autouse=True)
def _clean(monkeypatch):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    for v in ("SGEMM_GB300_PERSIST", "SGEMM_GB300_STREAM_K", "SGEMM_GB300_PAIR", "SGEMM_GB300_TILE_N",
              "SGEMM_GB300_SPLIT_K", "SGEMM_GB300_SPLIT_A_IN", "SGEMM_GB300_SPLIT_B_IN", "SGEMM_GB300_TRANS"):
        monkeypatch.delenv(v, raising=False)


def _run(p, exact=False):
    pl = Placed(p)
    st = pl.run(TC)
    assert st == 0, binding.status_string(st)
    C, guard_ok = pl.result()
    assert guard_ok, "a write landed outside the m x n window of C"
    assert pl.inputs_untouched()
    ok, worst, where = check_full(p, C, exact=exact)
    assert ok, f"worst |C - r| / tol = {worst} at {where}"
    assert binding.device_status() == 0
    return C


@pytest.mark.parametrize("m,n,k,lda,env", [
    (2176, 2304, 512, None, {}),                                  # 153 tiles: CTA 0 takes two
    (3000, 2600, 300, None, {}),                                  # ragged, 1-2 tiles per CTA
    (5000, 1100, 777, 777, {}),                                   # A in row phases
    (2600, 2000, 300, None, {"SGEMM_GB300_TILE_N": "128"}),       # 128-wide tiles
    (40000, 128, 256, None, {"SGEMM_GB300_STREAM_K": "0", "SGEMM_GB300_TRANS": "1"}),   # transposed tiles
])
def test_persistent_matches_oracle_and_one_cta_per_tile(monkeypatch, m, n, k, lda, env):
    for key, val in env.items():
        monkeypatch.setenv(key, val)
    p = inputs.make_problem(m, n, k, alpha=1.25, beta=-0.5, seed=m + k, a="normal", b="uniform", c="uniform",
                            lda=lda)
    st, plan = binding.plan(p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, path=TC)
    assert st == 0 and plan["persistent"] == 1 and plan["tiles"] > plan["grid"], plan
    C1 = _run(p)
    monkeypatch.setenv("SGEMM_GB300_PERSIST", "0")
    st, plan = binding.plan(p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, path=TC)
    assert plan["persistent"] == 0
    C0 = _run(p)
    assert (C1 == C0).all()


def test_persistent_integer_twin_bit_exact():
    p = inputs.make_problem(3000, 2600, 500, alpha=2.0, beta=0.5, seed=3, a="int", b="int", c="int")
    st, plan = binding.plan(p.m, p.n, p.k, p.alpha, 256, p.lda, 256, p.ldb, p.beta, 256, p.ldc, path=TC)
    assert plan["persistent"] == 1
    _run(p, exact=True)
