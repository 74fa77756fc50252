"""Pins of the FP64 sum oracle (CPU): closed forms, exact integer sums, a
library cross-check, the tolerance formula, and planted mistakes."""
import numpy as np
import pytest
import torch

import oracle


def pin_closed_form(f):
    """sum of 1..N = N(N+1)/2 (every value and partial sum exact)."""
    for N in (1, 2, 7, 1000, 4097, 1 << 20):
        x = np.arange(1, N + 1, dtype=np.float32)
        s, a = f(x)
        if s != N * (N + 1) / 2 or a != s:
            return False
        s, a = f(-x)
        if s != -N * (N + 1) / 2 or a != N * (N + 1) / 2:
            return False
    return True


def pin_integers(f):
    rng = np.random.default_rng(1)
    for n in (0, 1, 5, 999, 100003):
        x = rng.integers(-1000, 1001, size=n).astype(np.float32)
        s, a = f(x)
        if s != sum(int(v) for v in x) or a != sum(abs(int(v)) for v in x):
            return False
    return True


def pin_library(f):
    rng = np.random.default_rng(2)
    x = rng.standard_normal(300001).astype(np.float32)
    s, a = f(x)
    t = torch.from_numpy(x).double()
    return abs(s - t.sum().item()) <= 1e-12 * t.abs().sum().item() and abs(a - t.abs().sum().item()) <= 1e-12 * a


PINS = [pin_closed_form, pin_integers, pin_library]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_sum_oracle_passes_pin(pin):
    assert pin(oracle.sum_f64)


def _loop(x, drop_last=False, double_first=False, no_abs=False):
    x = [float(v) for v in np.asarray(x, np.float32).reshape(-1)]
    if drop_last and x:
        x = x[:-1]
    if double_first and x:
        x = [x[0]] + x
    return sum(x), sum(v if no_abs else abs(v) for v in x)


@pytest.mark.parametrize("kw", [dict(drop_last=True), dict(double_first=True), dict(no_abs=True)],
                         ids=["drop_last", "double_first", "no_abs"])
def test_pins_reject_planted_mistake(kw):
    assert not all(p(lambda x: _loop(x, **kw)) for p in (pin_closed_form, pin_integers))


def test_unmutated_loop_passes():
    assert pin_closed_form(_loop) and pin_integers(_loop)


def test_sum_tolerance_formula():
    # gamma_1 = u / (1 - u): a single rounding
    u = 2.0 ** -24
    assert oracle.sum_tolerance(1.0, 1) == u / (1 - u)
    assert oracle.sum_within_tolerance(1.0 + 0.5 * u, 1.0, 1.0, 1)
    assert not oracle.sum_within_tolerance(1.0 + 2 * u, 1.0, 1.0, 1)
    assert not oracle.sum_within_tolerance(float("nan"), 1.0, 1.0, 10)


def test_tree_depth_of_three_launches_by_hand():
    """Depths worked out by hand from the launch shape the header states.
    2^28 aligned values on 152 SMs: min(2^28 / 8192, 4 * 152) = 608 blocks,
    608 * 512 = 311296 threads; 2^26 float4 loads over them is 215.6, so a
    thread's accumulator takes 216 values, no tail; 216 + 2 + 5 + 5 + 608 =
    836.  4099 values, 4-byte loads: one block of 512 threads, 9 values per
    thread (4099 / 512 = 8.006), 9 + 12 + 1 = 22.  5 aligned values: one
    block, one float4 and the one-value tail in thread 0's first
    accumulator, 2 + 12 + 1 = 15."""
    import reduce_model
    assert reduce_model.tree_depth(1 << 28, 152, vec=True) == 836
    assert reduce_model.tree_depth(4099, 152, vec=False) == 22
    assert reduce_model.tree_depth(5, 152, vec=True) == 15


def test_reduce_model_matches_the_header():
    """The launch constants the depth model assumes are the ones the header
    declares (a change of the kernel's launch shape must change both)."""
    import os
    import re
    import reduce_model
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    text = open(os.path.join(root, "include", "sgemm_gb300.h")).read()
    got = dict(re.findall(r"#define (SGEMM_REDUCE_\w+) (\d+)", text))
    assert int(got["SGEMM_REDUCE_THREADS"]) == reduce_model.THREADS
    assert int(got["SGEMM_REDUCE_BLOCKS_PER_SM"]) == reduce_model.BLOCKS_PER_SM
