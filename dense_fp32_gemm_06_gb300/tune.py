"""Sweeps of the tensor-core path's plan choices for given shapes.

    python -m dense_fp32_gemm_06_gb300.tune --shapes 1000,1500,777 256,256,8192 ...
    python -m dense_fp32_gemm_06_gb300.tune --policy --shapes 2048,2048,2048 ...

For each shape the operands are split once; then the GEMM kernel alone
(``sgemm_tf32x3_split_gemm``) is timed with CUDA events, after an L2 flush,
for every tile width (256, 128) and split-K factor (1, 2, 3, 4, 6, 8)
pinned through the library's tuning variables ``SGEMM_GB300_TILE_N`` and
``SGEMM_GB300_SPLIT_K``, and once more with the library's own choice.  One
line per shape: the automatic choice's time, the best configuration, and
every configuration's median time in microseconds.

--policy: whole calls (sgemm, splits included) under each setting of the
plan's other choices -- stream-K (SGEMM_GB300_STREAM_K), the transposed
tile for n <= 128 (SGEMM_GB300_TRANS), A split inside the GEMM
(SGEMM_GB300_SPLIT_A_IN) -- and under the library's own plan.  The settings
take turns within each repetition (L2 flushed before every call, CUDA-event
timed) so that clock and power drift falls on all of them alike; one line
per shape with the plan the device made, every setting's median time, and
the plan of each setting that differs from it.
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


POLICY_VARS = ("SGEMM_GB300_STREAM_K", "SGEMM_GB300_TRANS", "SGEMM_GB300_SPLIT_A_IN")


def policy(m, n, k, reps=20):
    """({setting: median us}, {setting: plan}) of whole tensor-core calls;
    setting "auto" is the library's own plan, the others pin one tuning
    variable to 0 or 1."""
    import torch
    from . import binding
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(2 * L2_BYTES // 4, device="cuda")
    A = torch.randn(m, k, device="cuda")
    B = torch.randn(k, n, device="cuda")
    C = torch.zeros(m, n, device="cuda")

    def call():
        st = binding.sgemm_raw(m, n, k, 1.0, A.data_ptr(), k, B.data_ptr(), n, 0.0, C.data_ptr(), n,
                               stream.cuda_stream, binding.PATH_TF32X3)
        if st:
            raise RuntimeError(binding.status_string(st))

    def use(var, val):
        for v in POLICY_VARS:
            os.environ.pop(v, None)
        if var is not None:
            os.environ[var] = val

    settings = [("auto", None, None)]
    for var in POLICY_VARS:
        if var == "SGEMM_GB300_TRANS" and n > 128:
            continue
        settings += [(f"{var[12:].lower()}={val}", var, val) for val in ("0", "1")]
    saved = {v: os.environ.get(v) for v in POLICY_VARS}
    times, plans = {name: [] for name, _, _ in settings}, {}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        for name, var, val in settings:
            use(var, val)
            st, pl = binding.plan(m, n, k, 1.0, A.data_ptr(), k, B.data_ptr(), n, 0.0, C.data_ptr(), n,
                                  path=binding.PATH_TF32X3, num_sms=0)
            plans[name] = pl
            for _ in range(3):
                call()
        for _ in range(reps):
            for name, var, val in settings:
                use(var, val)
                flush_buf.fill_(1.0)
                e0.record(stream)
                call()
                e1.record(stream)
                e1.synchronize()
                times[name].append(e0.elapsed_time(e1) * 1e3)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    return {name: statistics.median(ts) for name, ts in times.items()}, plans


def plan_text(pl):
    t = f"{pl['bm']}x{pl['bn']}"
    if pl["trans"]:
        t += " transposed"
    if pl["stream_k"]:
        t += " stream-K"
    elif pl["split_k"] > 1:
        t += f" split-K {pl['split_k']}"
    t += ", A split " + ("in the GEMM" if pl["a_in_kernel"] else "pass (lo only)" if pl["a_lo_only"] else "pass")
    return t


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
    ap.add_argument("--policy", action="store_true", help="whole calls under each plan choice (see above)")
    args = ap.parse_args(argv)
    if args.policy:
        for spec in args.shapes:
            m, n, k = (int(x) for x in spec.split(","))
            res, plans = policy(m, n, k, reps=args.reps)
            best = min(res, key=res.get)
            cells = " ".join(f"{name}:{us:.1f}" + ("" if plans[name] == plans["auto"] else
                                                   f"[{plan_text(plans[name])}]") for name, us in res.items())
            print(f"{(m, n, k)} auto={res['auto']:.1f}us [{plan_text(plans['auto'])}] best={best} "
                  f"{2 * m * n * k / res[best] / 1e6:.1f}TF | {cells}", flush=True)
        return
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
