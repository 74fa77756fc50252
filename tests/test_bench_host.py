"""Host-side logic of bench.py that needs no GPU: the multi-rank reduction
(two gloo ranks on CPU), the reference arm's rank handling and JSON line,
and the TFLOPS formula against the figures the pages print."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from dense_fp32_gemm_06_gb300 import inputs  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(values[rank], world)
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    """The timed region is the slowest rank's: every rank gets the max."""
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    values = [12.5, 17.25]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(out.get(timeout=5) for _ in range(2))
    assert got == {0: 17.25, 1: 17.25}


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5


def _run_bench(args, env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_without_work():
    r = _run_bench(["--impl", "reference", "--workload", "256^3", "--steps", "1", "--warmup", "0"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_json_line():
    r = _run_bench(["--impl", "reference", "--workload", "256^3", "--steps", "2", "--warmup", "1"],
                   {"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOPS"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_tflops_formula_reproduces_the_pages_figures():
    """TFLOPS = 2mnk x launches / seconds reproduces the four 2048^3 figures
    printed on blog.lightlisten.com "gemm优化" (section 最终结果)."""
    with open(os.path.join(ROOT, "tests", "golden", "timings_2048.json")) as fh:
        g = json.load(fh)
    p = inputs.Problem(2048, 2048, 2048, 1.0, 0.0, None, None, None, 2048, 2048, 2048, 0, ())
    for row in g["rows"]:
        got = bench.tflops(p, row["ms"], g["inputs"]["launches"])
        assert round(got, 3) == pytest.approx(row["tflops"], abs=1e-3), row


def test_workload_names_match_the_generator():
    assert set(bench.WORKLOAD_TEXT) == set(inputs.WORKLOADS)
    args = bench.parse(["--workload", "1000x1500x777"])
    p, text = bench.load_problem(args)
    assert (p.m, p.n, p.k, p.lda) == (1000, 1500, 777, 777) and "1000x1500x777" in text


def test_traffic_record_matches_size_and_sources(tmp_path, monkeypatch):
    """The ncu DRAM figure is reported only for the size it was captured on
    and only while the kernel's sources are unchanged."""
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    h = bench.kernel_source_hash("tf32x3_raw_ab")
    recs = {"tf32x3_raw_ab": [{"units": 10, "source_hash": h, "dram_bytes_per_launch": 111},
                            {"units": 20, "source_hash": "stale", "dram_bytes_per_launch": 222}],
            "ffma": {"units": 30, "source_hash": bench.kernel_source_hash("ffma"), "dram_bytes_per_launch": 333}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(recs))
    assert bench.traffic_record("tf32x3_raw_ab", 10) == 111
    assert bench.traffic_record("tf32x3_raw_ab", 20) is None      # sources changed since the capture
    assert bench.traffic_record("tf32x3_raw_ab", 30) is None      # never captured at this size
    assert bench.traffic_record("ffma", 30) == 333              # single-record form
    assert bench.traffic_record("tf32x3_presplit", 10) is None


def test_kernel_hash_ignores_comments_only():
    """A traffic figure is void once the kernel's code changes, not when only
    its comments do."""
    code = "int f(int x) {\n    return x + 1;   // one more\n}\n/* a note */\n"
    assert bench.strip_comments(code) == bench.strip_comments(code.replace("one more", "plus one"))
    assert bench.strip_comments(code) != bench.strip_comments(code.replace("x + 1", "x + 2"))
    assert "note" not in bench.strip_comments(code) and "return x + 1;" in bench.strip_comments(code)


def test_kernel_hash_covers_the_planner(tmp_path, monkeypatch):
    """The plan (tiles, raster groups, schedule) sets the launch whose
    traffic a record holds, so a change to the planner's code voids every
    family's records too."""
    import shutil
    src = os.path.join(bench.ROOT, "dense_fp32_gemm_06_gb300", "csrc")
    dst = tmp_path / "dense_fp32_gemm_06_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = {f: bench.kernel_source_hash(f) for f in bench.KERNEL_SOURCES}
    planner = dst / "sgemm_api.cu"
    planner.write_text(planner.read_text() + "\nstatic int another_plan_constant = 1;\n")
    after = {f: bench.kernel_source_hash(f) for f in bench.KERNEL_SOURCES}
    assert all(before[f] != after[f] for f in before)
