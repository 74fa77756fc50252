"""The seeded input generator shared by the CUDA path's tests and the
oracle: splitmix64 against its published output sequence and against the
sequential stream (any slice drawn without its prefix), the value maps of
each distribution, and determinism of whole problems."""
import numpy as np

from dense_fp32_gemm_06_gb300 import inputs

# the first five outputs of splitmix64 seeded with 0 (the reference
# generator of Steele, Lea and Flood as distributed in Vigna's splitmix64.c)
SEED0 = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC, 0x1B39896A51A8749B]


def _sequential(seed, count):
    """The sequential stream, one 64-bit step at a time (Python integers)."""
    mask = (1 << 64) - 1
    state, out = seed, []
    for _ in range(count):
        state = (state + 0x9E3779B97F4A7C15) & mask
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_known_answer():
    assert [int(x) for x in inputs.splitmix64(0, 0, 5)] == SEED0


def test_splitmix64_slices_are_the_sequential_stream():
    for seed in (0, 1, 3, 12345, (1 << 63) + 17):
        seq = _sequential(seed, 300)
        for start, count in ((0, 300), (1, 7), (17, 64), (250, 50)):
            assert [int(x) for x in inputs.splitmix64(seed, start, count)] == seq[start:start + count]


def test_uniform_and_integer_maps():
    u = inputs.draw_matrix("uniform", 5, 0, 300, 400)
    assert u.dtype == np.float32 and u.min() >= -1.0 and u.max() < 1.0
    # 2 * (24-bit fraction) - 1: every value is a multiple of 2^-23
    assert np.all(np.mod(u.astype(np.float64) * 2.0 ** 23, 1.0) == 0.0)
    assert abs(float(u.mean())) < 0.01 and abs(float(u.var()) - 1.0 / 3.0) < 0.01
    u01 = inputs.draw_matrix("uniform01", 5, 0, 300, 400)
    assert u01.min() >= 0.0 and u01.max() < 1.0
    np.testing.assert_array_equal(u, 2.0 * u01 - 1.0)   # the same draws, the same u
    t = inputs.draw_matrix("int", 5, 0, 300, 400)
    assert set(np.unique(t).tolist()) == set(range(-4, 5))
    np.testing.assert_array_equal(t, np.floor(9.0 * u01.astype(np.float64)) - 4.0)


def test_normal_moments():
    z = inputs.draw_matrix("normal", 9, 0, 500, 400).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert np.isfinite(z).all() and np.abs(z).max() < 7.0


def test_problems_are_deterministic_and_seed_dependent():
    a = inputs.make_problem(64, 48, 40, alpha=1.5, beta=0.5, seed=3, a="normal", b="uniform", c="int")
    b = inputs.make_problem(64, 48, 40, alpha=1.5, beta=0.5, seed=3, a="normal", b="uniform", c="int")
    c = inputs.make_problem(64, 48, 40, alpha=1.5, beta=0.5, seed=4, a="normal", b="uniform", c="int")
    for x, y in ((a.A, b.A), (a.B, b.B), (a.C0, b.C0)):
        np.testing.assert_array_equal(x, y)
    assert not np.array_equal(a.A, c.A)
