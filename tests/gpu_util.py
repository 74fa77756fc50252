"""Helpers for the GPU parity tests: place a synthetic problem in device
memory (optionally misaligned and with guard bands), run the C ABI, and
compare against the FP64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dense_fp32_gemm_06_gb300 import binding

SENTINEL = np.float32(-7777.25)


class Placed:
    """A problem copied to the GPU.  Each operand lives in a flat buffer at
    element offset ``off`` (so ``off % 4 != 0`` misaligns it), followed and
    preceded by sentinel values that must survive the call."""

    def __init__(self, p, off=(0, 0, 0), guard=64):
        self.p = p
        self.off = off
        self.guard = guard
        self.bufs = []
        for arr, o, rows, cols, ld in ((p.A, off[0], p.m, p.k, p.lda), (p.B, off[1], p.k, p.n, p.ldb),
                                       (p.C0, off[2], p.m, p.n, p.ldc)):
            span = (rows - 1) * ld + cols if rows > 0 and cols > 0 else 0
            host = np.full(guard + o + max(span, 1) + guard, SENTINEL, dtype=np.float32)
            if span:
                flat = np.ascontiguousarray(arr).reshape(-1)[:span]
                host[guard + o: guard + o + span] = flat
            self.bufs.append((torch.from_numpy(host).cuda(), guard + o, span, rows, cols, ld))

    def ptr(self, i):
        buf, start, _, _, _, _ = self.bufs[i]
        return buf.data_ptr() + 4 * start

    def run(self, path=binding.PATH_AUTO, alpha=None, beta=None):
        p = self.p
        st = binding.sgemm_raw(p.m, p.n, p.k, p.alpha if alpha is None else alpha, self.ptr(0), p.lda,
                               self.ptr(1), p.ldb, p.beta if beta is None else beta, self.ptr(2), p.ldc,
                               torch.cuda.current_stream().cuda_stream, path)
        torch.cuda.synchronize()
        return st

    def result(self):
        """(C as m x n float32, guard_ok): guard_ok is False when any element
        outside the m x n window of C (guards, row gaps) changed."""
        buf, start, span, rows, cols, ld = self.bufs[2]
        host = buf.cpu().numpy()
        ok = bool(np.all(host[:start] == SENTINEL) and np.all(host[start + span:] == SENTINEL))
        if span:
            win = np.full(rows * ld, SENTINEL, dtype=np.float32)
            win[:span] = host[start:start + span]
            win = win.reshape(rows, ld)
            # the gaps between rows (ld > cols) hold the generator's padding
            # (NaN) for C0 and must be untouched; the last row has no gap
            # inside the span (what follows it is the sentinel guard above)
            gaps = win[:rows - 1, cols:]
            if ld > cols:
                orig = np.ascontiguousarray(self.p.C0).reshape(rows, ld)[:rows - 1, cols:]
                same = (gaps == orig) | (np.isnan(gaps) & np.isnan(orig))
                ok = ok and bool(np.all(same))
            return np.ascontiguousarray(win[:, :cols]), ok
        return np.zeros((rows, cols), np.float32), ok

    def inputs_untouched(self):
        for i, (arr, o) in enumerate(((self.p.A, self.off[0]), (self.p.B, self.off[1]))):
            buf, start, span, rows, cols, ld = self.bufs[i]
            host = buf.cpu().numpy()
            want = np.full_like(host, SENTINEL)
            if span:
                want[start:start + span] = np.ascontiguousarray(arr).reshape(-1)[:span]
            if not np.array_equal(host.view(np.uint32), want.view(np.uint32)):
                return False
        return True


def check_full(p, C, exact=False):
    """Compares C with the oracle on every element.  exact=True demands
    float equality (integer twins); returns (ok, worst_ratio, where)."""
    R, E, Rf = oracle.problem_f64(p)
    if exact:
        bad = ~(C == Rf)
        if np.any(bad):
            idx = np.argwhere(bad)[0]
            return False, float("inf"), tuple(idx)
        return True, 0.0, None
    C0v = p.C0[:, :p.n] if p.beta != 0.0 else None
    return oracle.within_tolerance(C, R, E, p.beta, C0v)


def check_sampled(p, C, rows, cols, exact=False):
    R, E = oracle.problem_f64_sampled(p, rows, cols)
    got = C[rows, cols]
    if exact:
        ok = bool(np.all(got.astype(np.float64) == R))
        return ok, 0.0 if ok else float("inf"), None
    C0v = p.C0[rows, cols] if p.beta != 0.0 else None
    return oracle.within_tolerance(got, R, E, p.beta, C0v)


def projection_ratios(A, B, C0, C, alpha, beta, seed):
    """Freivalds' check of every output of C = alpha A B + beta C0 at once,
    in FP64 on the tensors' device: (max over rows of |C x - ref| / bound,
    max over columns of |y^T C - ref| / bound) for Gaussian x, y drawn from
    `seed`.  The bound of a row (column) is the sum over it of the
    per-element FP32 bound 1e-5 |alpha| sum_t |A_it||B_tj| + 1e-6 |beta C0_ij|
    (against |x_j|, |y_i|), so a C within that bound everywhere gives ratios
    <= 1.  C0 is not used when beta = 0."""
    g = torch.Generator(device=C.device).manual_seed(seed)
    m, n = C.shape
    x = torch.randn(n, 1, device=C.device, dtype=torch.float64, generator=g)
    y = torch.randn(1, m, device=C.device, dtype=torch.float64, generator=g)
    Ad, Bd, Cd = A.double(), B.double(), C.double()
    ref_x = alpha * (Ad @ (Bd @ x))
    tol_x = 1e-5 * abs(alpha) * (Ad.abs() @ (Bd.abs() @ x.abs()))
    ref_y = alpha * ((y @ Ad) @ Bd)
    tol_y = 1e-5 * abs(alpha) * ((y.abs() @ Ad.abs()) @ Bd.abs())
    if beta != 0:
        C0d = C0.double()
        ref_x = ref_x + beta * (C0d @ x)
        tol_x = tol_x + 1e-6 * abs(beta) * (C0d.abs() @ x.abs())
        ref_y = ref_y + beta * (y @ C0d)
        tol_y = tol_y + 1e-6 * abs(beta) * (y.abs() @ C0d.abs())
    rx = ((Cd @ x - ref_x).abs() / tol_x).max().item()
    ry = ((y @ Cd - ref_y).abs() / tol_y).max().item()
    return rx, ry
