"""Tile-width x split-K sweep of the tensor-core GEMM for given shapes.

    python -m dense_fp32_gemm_06_gb300.tune --shapes 1000,1500,777 256,256,8192 ...

For each shape the operands are split once; then the GEMM kernel alone
(``sgemm_tf32x3_split_gemm``) is timed with CUDA events, after an L2 flush,
for every tile width (256, 128) and split-K factor (1, 2, 3, 4, 6, 8)
pinned through the library's tuning variables ``SGEMM_GB300_TILE_N`` and
``SGEMM_GB300_SPLIT_K``, and once more with the library's own choice.  One
line per shape: the automatic choice's time, the best configuration, and
every configuration's median time in microseconds.
"""
from __future__ import annotations

import argparse
import itertools
import os
import statistics

L2_BYTES = 129 * 2 ** 20


def _median_us(fn, flush, stream, reps):
    import torch
    ts = []
    for _ in range(reps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    return statistics.median(ts)


def sweep(m, n, k, reps=20, widths=(256, 128), splits=(1, 2, 3, 4, 6, 8), max_ctas=8 * 152):
    import torch
    from . import binding
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(2 * L2_BYTES // 4, device="cuda")
    A = torch.randn(m, k, device="cuda")
    B = torch.randn(k, n, device="cuda")
    C = torch.zeros(m, n, device="cuda")
    ka = binding.ka_of(k)
    ah, al = torch.empty(m * ka, device="cuda"), torch.empty(m * ka, device="cuda")
    bh, bl = torch.empty(n * ka, device="cuda"), torch.empty(n * ka, device="cuda")
    binding.tf32x3_split_a(A, ah, al)
    binding.tf32x3_split_b(B, bh, bl)

    def gemm():
        st = binding.tf32x3_split_gemm_raw(m, n, k, 1.0, ah.data_ptr(), al.data_ptr(), bh.data_ptr(),
                                           bl.data_ptr(), 0.0, C.data_ptr(), n, stream.cuda_stream)
        if st:
            raise RuntimeError(binding.status_string(st))

    flush = lambda: flush_buf.fill_(1.0)  # noqa: E731
    saved = {v: os.environ.get(v) for v in ("SGEMM_GB300_TILE_N", "SGEMM_GB300_SPLIT_K")}
    results = {}
    try:
        for bn, s in itertools.product(widths, splits):
            if bn == 256 and n <= 128:
                continue
            os.environ["SGEMM_GB300_TILE_N"] = str(bn)
            os.environ["SGEMM_GB300_SPLIT_K"] = str(s)
            st, pl = binding.plan(m, n, k, lda=k, path=binding.PATH_TF32X3)
            if st or pl["grid"] > max_ctas:
                continue
            for _ in range(3):
                gemm()
            results[(bn, s)] = _median_us(gemm, flush, stream, reps)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    for _ in range(3):
        gemm()
    auto = _median_us(gemm, flush, stream, reps)
    return auto, results


def reduce_bandwidth(n=1 << 28, reps=50):
    """GB/s of reduce_sum_f32 on n floats (4n bytes read per call), CUDA
    events, median of `reps` calls (n = 2^28: 1 GiB, far larger than L2)."""
    import torch
    from . import binding
    x = torch.empty(n, device="cuda").uniform_(-1, 1)
    out = torch.empty(1, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(3):
        binding.reduce_sum(x, out)
    us = _median_us(lambda: binding.reduce_sum(x, out), lambda: None, stream, reps)
    return 4.0 * n / (us * 1e-6) / 1e9, us


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--shapes", nargs="+", default=["1000,1500,777", "256,256,8192", "300,700,5000",
                                                    "129,257,4096", "2048,2048,2048", "16384,128,8192",
                                                    "500,500,300", "4096,4096,1024", "1024,1024,16384",
                                                    "2048,1024,8192"])
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--reduce", type=int, default=0, help="measure reduce_sum_f32 on this many floats instead")
    args = ap.parse_args(argv)
    if args.reduce:
        gbs, us = reduce_bandwidth(args.reduce)
        print(f"reduce_sum_f32 n={args.reduce} {us:.1f} us {gbs:.1f} GB/s", flush=True)
        return
    for spec in args.shapes:
        m, n, k = (int(x) for x in spec.split(","))
        auto, res = sweep(m, n, k, reps=args.reps)
        (bbn, bs), bus = min(res.items(), key=lambda kv: kv[1])
        cells = " ".join(f"{bn}/{s}:{us:.0f}" for (bn, s), us in sorted(res.items()))
        print(f"{(m, n, k)} auto={auto:.0f}us best={bbn}/{bs}:{bus:.0f}us "
              f"{2 * m * n * k / bus / 1e6:.1f}TF | {cells}", flush=True)


if __name__ == "__main__":
    main()
