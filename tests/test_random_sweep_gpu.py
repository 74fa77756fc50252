"""A seeded random sweep over the whole call: shapes from 1 to a few
thousand on each side, padded leading dimensions, misaligned bases, random
alpha and beta (beta = 0 over a NaN-filled C), both paths and AUTO, and the
library's tuning pins (stream-K, CTA pairs, split passes, tile widths, the
FFMA per-thread tile) -- each call against the FP64 oracle on every output
(integer twins bit for bit), with guard bands around C and A, B unwritten."""
import numpy as np
import pytest
import torch

from dense_fp32_gemm_06_gb300 import binding, inputs
from gpu_util import Placed, check_full

pytestmark = pytest.mark.gpu

PINS = [{}, {}, {}, {"SGEMM_GB300_STREAM_K": "1"}, {"SGEMM_GB300_PAIR": "1"},
        {"SGEMM_GB300_SPLIT_A_IN": "0", "SGEMM_GB300_SPLIT_B_IN": "0"}, {"SGEMM_GB300_SPLIT_B_IN": "1"},
        {"SGEMM_GB300_TILE_N": "128"}, {"SGEMM_GB300_FFMA_RN": "16"}, {"SGEMM_GB300_SPLIT_K": "2"}]
KEYS = sorted({k for pin in PINS for k in pin})


def _cases(count=48, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        m, n, k = (int(rng.choice([rng.integers(1, 300), rng.integers(1, 2500)])) for _ in range(3))
        if m * n * k > 1.5e8:
            continue
        out.append(dict(m=m, n=n, k=k, lda=k + int(rng.choice([0, 0, 1, 3, 4])), ldb=n + int(rng.choice([0, 0, 2, 4])),
                        ldc=n + int(rng.choice([0, 0, 1])), offs=tuple(int(rng.choice([0, 0, 1, 3])) for _ in range(3)),
                        alpha=float(rng.choice([1.0, -0.5, 2.0, 0.75])), beta=float(rng.choice([0.0, 0.0, 1.0, -1.5])),
                        twin=bool(rng.integers(0, 2)), path=int(rng.choice([binding.PATH_AUTO, binding.PATH_FFMA,
                                                                                binding.PATH_TF32X3])),
                        pin=PINS[int(rng.integers(0, len(PINS)))], seed=int(rng.integers(0, 1 << 30))))
    return out


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"{c['m']}x{c['n']}x{c['k']}")
def test_random_call_matches_oracle(monkeypatch, case):
    for key in KEYS:
        monkeypatch.delenv(key, raising=False)
    for key, val in case["pin"].items():
        monkeypatch.setenv(key, val)
    twin = case["twin"]
    dist = "int" if twin else "normal"
    p = inputs.make_problem(case["m"], case["n"], case["k"], alpha=case["alpha"], beta=case["beta"], seed=case["seed"],
                            a=dist, b="int" if twin else "uniform", c=("int" if twin else "uniform") if case["beta"] else None,
                            lda=case["lda"], ldb=case["ldb"], ldc=case["ldc"], c_fill=float("nan"))
    pl = Placed(p, off=case["offs"])
    st = pl.run(case["path"])
    assert st == 0, binding.status_string(st)
    C, guard_ok = pl.result()
    assert guard_ok, "a write landed outside the m x n window of C"
    assert pl.inputs_untouched(), "A or B was modified"
    ok, worst, where = check_full(p, C, exact=twin)
    assert ok, f"worst |C - r| / tol = {worst} at {where}"
    assert binding.device_status() == 0
