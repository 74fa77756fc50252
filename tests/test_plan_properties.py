"""Invariants of the launch plan over many seeded random problems (host
only, a 152-SM device): the tiles cover the output, the grid and thread
counts agree with the tile and split choices, shared memory fits a CTA, and
the operand sources obey the rules the kernels rely on (an operand read by
TMA as stored has a 16-byte aligned base and 16-byte rows; an A read in row
phases is K-major on untransposed single-CTA tiles; CTA pairs read A by
TMA; stream-K and split-K exclude each other; transposed tiles only for
n <= 128)."""
import numpy as np

from dense_fp32_gemm_06_gb300 import binding

SMEM_MAX = 227 * 1024
SMS = 152


def _draw(rng):
    pick = rng.integers(0, 4)
    if pick == 0:
        m, n, k = (int(x) for x in rng.integers(1, 300, 3))
    elif pick == 1:
        m, n, k = (int(x) for x in rng.integers(1, 5000, 3))
    elif pick == 2:
        m, n, k = int(rng.integers(1, 20000)), int(rng.integers(1, 160)), int(rng.integers(1, 10000))
    else:
        m, n, k = (int(2 ** rng.integers(0, 14)) + int(rng.integers(-1, 2)) for _ in range(3))
    m, n, k = max(m, 1), max(n, 1), max(k, 1)
    lda = k + int(rng.choice([0, 0, 1, 2, 3, 4, 17]))
    ldb = n + int(rng.choice([0, 0, 1, 2, 3, 4, 17]))
    ldc = n + int(rng.choice([0, 0, 1, 4]))
    a_ptr = 256 + 4 * int(rng.choice([0, 0, 0, 1, 2, 3]))
    b_ptr = 4096 + 4 * int(rng.choice([0, 0, 0, 1, 2, 3]))
    c_ptr = 65536 + 4 * int(rng.choice([0, 0, 1]))
    path = int(rng.choice([binding.PATH_AUTO, binding.PATH_FFMA, binding.PATH_TF32X3]))
    return m, n, k, lda, ldb, ldc, a_ptr, b_ptr, c_ptr, path


def _ceil(a, b):
    return -(-a // b)


def test_plan_invariants_over_random_problems(monkeypatch):
    rng = np.random.default_rng(20261202)
    seen = {"ffma": 0, "tc": 0, "pair": 0, "trans": 0, "sk": 0, "split": 0, "phased": 0, "persistent": 0}
    for i in range(3600):
        # the last 600 with CTA pairs requested (the default takes them only
        # for one wave of 256 x 256 tiles)
        if i == 3000:
            monkeypatch.setenv("SGEMM_GB300_PAIR", "1")
        m, n, k, lda, ldb, ldc, ap, bp, cp, path = _draw(rng)
        st, p = binding.plan(m, n, k, 1.0, ap, lda, bp, ldb, 0.5, cp, ldc, path=path, num_sms=SMS)
        assert st == 0, (m, n, k, lda, ldb, ldc, ap, bp, cp, path, st)
        where = (m, n, k, lda, ldb, ap, bp, path, p)
        assert 0 < p["smem_bytes"] <= SMEM_MAX, where
        if p["kernel"] == 0:                      # FFMA
            seen["ffma"] += 1
            assert p["path"] == binding.PATH_FFMA or path == binding.PATH_AUTO, where
            assert p["tiles"] == _ceil(m, p["bm"]) * _ceil(n, p["bn"]) == p["grid"], where
            assert p["threads"] == (p["bm"] // (8 * p["rm"])) * (p["bn"] // (4 * p["rn"])) * 32, where
            assert p["k_tiles"] == _ceil(k, p["bk"]), where
            continue
        assert p["kernel"] == 2, where           # tensor core (alpha != 0, k > 0)
        seen["tc"] += 1
        assert p["threads"] == 384, where
        a_tma = ap % 16 == 0 and lda % 4 == 0
        b_tma = bp % 16 == 0 and ldb % 4 == 0
        if p["b_in_kernel"]:
            assert b_tma, where
        if p["a_in_kernel"] and not a_tma:       # A read in row phases
            seen["phased"] += 1
            assert not p["trans"] and not p["pair"], where
        if p["pair"]:
            seen["pair"] += 1
            assert (p["bm"], p["bn"]) == (256, 256) and p["split_k"] == 1 and p["stream_k"] == 0, where
            assert not p["persistent"], where
            assert p["grid"] == 2 * p["tiles"] == 2 * _ceil(m, 256) * _ceil(n, 256), where
            continue
        if p["trans"]:
            seen["trans"] += 1
            assert n <= 128 and (p["bm"], p["bn"]) == (256, 128), where
        else:
            assert p["bm"] == 128 and p["bn"] in (128, 256), where
        assert p["tiles"] == _ceil(m, p["bm"]) * _ceil(n, p["bn"]), where
        assert 1 <= p["split_k"] <= 8, where
        if p["stream_k"]:
            seen["sk"] += 1
            assert p["split_k"] == 1 and p["grid"] == p["stream_k"] == SMS and not p["persistent"], where
        elif p["persistent"]:
            seen["persistent"] += 1
            assert p["split_k"] == 1 and p["grid"] == SMS < p["tiles"], where
        else:
            assert p["grid"] == p["tiles"] * p["split_k"] and p["tiles"] * p["split_k"] <= SMS or p["split_k"] == 1, where
        if p["split_k"] > 1:
            seen["split"] += 1
            assert p["k_tiles"] // p["split_k"] >= 4, where
    # the draw reaches every kind of plan
    assert all(v > 0 for v in seen.values()), seen
