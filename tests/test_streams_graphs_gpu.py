"""Calls of the regular entry point on several streams at once do not
interfere (each takes its scratch and stream-K workspace from the pool in
stream order), and a call captured into a CUDA graph replays correctly
(the pool allocation, the stream-K counter reset, cluster launches and the
dependent launch of the GEMM become graph nodes).  The library's one-time
per-device set-up happens in a call before the capture."""
import numpy as np
import pytest
import torch

import oracle
from dense_fp32_gemm_06_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

TC = binding.PATH_TF32X3


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


# (m, n, k, beta, tuning variables): whole tiles, stream-K, transposed
# stream-K tiles, a split-K cluster, the FFMA path
PROBLEMS = [
    (2048, 2048, 256, 0.0, {}),
    (1000, 1500, 780, 0.5, {"SGEMM_GB300_STREAM_K": "1"}),
    (3000, 100, 2048, 1.0, {"SGEMM_GB300_STREAM_K": "1", "SGEMM_GB300_TRANS": "1"}),
    (300, 700, 5000, 0.0, {"SGEMM_GB300_STREAM_K": "0"}),
]


def _dev(p):
    return (torch.from_numpy(np.ascontiguousarray(p.A)).cuda(), torch.from_numpy(np.ascontiguousarray(p.B)).cuda(),
            torch.from_numpy(np.ascontiguousarray(p.C0)).cuda())


def _call(p, A, B, C, stream, path=TC):
    st = binding.sgemm_raw(p.m, p.n, p.k, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta, C.data_ptr(),
                           p.ldc, stream.cuda_stream, path)
    assert st == 0, binding.status_string(st)


def test_concurrent_streams_do_not_interfere(monkeypatch):
    probs = [inputs.make_problem(m, n, k, alpha=1.25, beta=beta, seed=i + 1, a="normal", b="uniform",
                                 c="uniform" if beta else None) for i, (m, n, k, beta, _) in enumerate(PROBLEMS)]
    # each problem alone, its tuning variables set only while it is planned
    refs = []
    for p, (_, _, _, _, env) in zip(probs, PROBLEMS):
        for key, val in env.items():
            monkeypatch.setenv(key, val)
        A, B, C = _dev(p)
        s = torch.cuda.current_stream()
        _call(p, A, B, C, s)
        torch.cuda.synchronize()
        refs.append(C.cpu().numpy())
        for key in env:
            monkeypatch.delenv(key)
    R, E, _ = oracle.problem_f64(probs[0])
    ok, worst, _ = oracle.within_tolerance(refs[0], R, E, 0.0, None)
    assert ok, worst
    # all of them at once, on four streams, three times over
    streams = [torch.cuda.Stream() for _ in probs]
    for _ in range(3):
        outs = []
        for p, s, (_, _, _, _, env) in zip(probs, streams, PROBLEMS):
            for key, val in env.items():
                monkeypatch.setenv(key, val)
            A, B, C = _dev(p)
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                _call(p, A, B, C, s)
            outs.append((A, B, C))
            for key in env:
                monkeypatch.delenv(key)
        torch.cuda.synchronize()
        for (A, B, C), ref in zip(outs, refs):
            assert np.array_equal(C.cpu().numpy(), ref)


@pytest.mark.parametrize("idx", range(len(PROBLEMS)))
def test_call_captured_in_a_cuda_graph(monkeypatch, idx):
    m, n, k, beta, env = PROBLEMS[idx]
    for key, val in env.items():
        monkeypatch.setenv(key, val)
    p = inputs.make_problem(m, n, k, alpha=1.5, beta=beta, seed=40 + idx, a="normal", b="uniform",
                            c="uniform" if beta else None)
    A, B, C = _dev(p)
    C0 = C.clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _call(p, A, B, C, s)   # one-time set-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    C.copy_(C0)
    with torch.cuda.graph(g, stream=s):
        _call(p, A, B, C, s)
    # replay on the captured inputs, then on new A values
    for rep in range(2):
        if rep == 1:
            p2 = inputs.make_problem(m, n, k, alpha=1.5, beta=beta, seed=90 + idx, a="normal", b="uniform",
                                     c="uniform" if beta else None)
            A.copy_(torch.from_numpy(np.ascontiguousarray(p2.A)))
            p = inputs.Problem(p.m, p.n, p.k, p.alpha, p.beta, p2.A, p.B, p.C0, p.lda, p.ldb, p.ldc, p.seed, p.dists)
        C.copy_(C0)
        g.replay()
        torch.cuda.synchronize()
        R, E, _ = oracle.problem_f64(p)
        ok, worst, where = oracle.within_tolerance(C.cpu().numpy()[:, :n], R, E, p.beta,
                                                   p.C0[:, :n] if p.beta != 0 else None)
        assert ok, f"replay {rep}: worst {worst} at {where}"
