"""Builds and loads the C-ABI CUDA library (in-tree, sm_103a only)."""
from __future__ import annotations

import ctypes
import os
import platform
import shutil
import subprocess
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
CSRC = os.path.join(_PKG, "csrc")
INCLUDE = os.path.join(_ROOT, "include")
LIB_DIR = os.path.join(_PKG, "_lib")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]
# the C ABI and planning, and the kernel units (compiled in parallel)
SOURCES = ["sgemm_api.cu", "tc_wide.cu", "tc_narrow.cu", "tc_trans.cu", "tc_pair.cu", "ffma.cu"]

_lock = threading.Lock()
_libs = {}


class SgemmError(RuntimeError):
    """A non-zero status from the C ABI, or a missing library."""

    def __init__(self, status: int, message: str):
        super().__init__(f"sgemm status {status}: {message}")
        self.status = status


def lib_path(checked: bool = False) -> str:
    """The release library, or (checked=True) the one compiled with
    SGEMM_GB300_CHECKED: every kernel index tested before its access."""
    kind = "checked_" if checked else ""
    return os.path.join(LIB_DIR, f"libsgemm_gb300_{kind}{platform.machine()}.so")


def _deps():
    out = [os.path.join(INCLUDE, "sgemm_gb300.h")]
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            out.append(os.path.join(CSRC, name))
    return out


def _stale(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in _deps())


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise SgemmError(-1, "nvcc not found: cannot build the CUDA library")


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compiles csrc/*.cu into one shared library for sm_103a; returns its
    path (the checked variant with checked=True)."""
    return build_all(force=force, verbose=verbose, variants=(checked,))[0]


def build_all(force: bool = False, verbose: bool = False, variants=(False, True)) -> list:
    """Compiles the release library and (variants containing True) the
    checked one, every object of every variant in parallel, then one link
    each.  Skips a variant whose library is newer than every source."""
    os.makedirs(LIB_DIR, exist_ok=True)
    cc = nvcc()
    jobs = []   # (target, objs, procs)
    for checked in variants:
        target = lib_path(checked)
        if not force and not _stale(target):
            jobs.append((target, None, []))
            continue
        obj_dir = os.path.join(LIB_DIR, f"obj_{'checked_' if checked else ''}{platform.machine()}")
        os.makedirs(obj_dir, exist_ok=True)
        objs, procs = [], []
        for src in SOURCES:
            obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
            objs.append(obj)
            cmd = [cc, *ARCH_FLAGS, *NVCC_FLAGS, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
            if checked:
                cmd.insert(1, "-DSGEMM_GB300_CHECKED")
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        jobs.append((target, objs, procs))
    out_paths = []
    for target, objs, procs in jobs:
        for cmd, p in procs:
            out, _ = p.communicate()
            if verbose or p.returncode:
                print(out.decode(errors="replace"))
            if p.returncode:
                raise SgemmError(-1, "nvcc failed: " + " ".join(cmd))
        if objs is not None:
            tmp = target + f".tmp{os.getpid()}"
            link = [cc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
            r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
            if r.returncode:
                print(r.stdout.decode(errors="replace"))
                raise SgemmError(-1, "nvcc link failed")
            os.replace(tmp, target)
        out_paths.append(target)
    return out_paths


# Exported symbols, in the order the header declares them.
EXPORTS = ["sgemm", "sgemm_ex", "sgemm_op", "sgemm_strided_batched", "sgemm_tf32x3_split_a", "sgemm_tf32x3_split_b", "sgemm_tf32x3_split_gemm",
           "sgemm_tf32x3_noalloc", "reduce_sum_f32", "sgemm_status_string", "sgemm_last_cuda_error", "sgemm_plan_for", "sgemm_device_status",
           "sgemm_selftest_wait", "sgemm_bounds_line", "sgemm_selftest_bounds", "sgemm_version"]


class Plan(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in (
        "path", "kernel", "bm", "bn", "bk", "rm", "rn", "threads", "stages", "grid", "tiles",
        "k_tiles", "smem_bytes", "b_vec", "c_vec", "group_m", "split_k", "op_a", "op_b", "a_vec",
        "a_in_kernel", "trans", "stream_k", "b_in_kernel", "pair", "persistent", "sk_parts")]


def _declare(lib):
    i, f, vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    gemm = [i, i, i, f, vp, i, vp, i, f, vp, i, vp]
    lib.sgemm.argtypes = gemm
    lib.sgemm.restype = i
    lib.sgemm_ex.argtypes = gemm + [i]
    lib.sgemm_ex.restype = i
    lib.sgemm_op.argtypes = [i, i] + gemm + [i]
    lib.sgemm_op.restype = i
    ll = ctypes.c_longlong
    lib.sgemm_strided_batched.argtypes = [i, i, i, i, i, f, vp, i, ll, vp, i, ll, f, vp, i, ll, i, vp, i]
    lib.sgemm_strided_batched.restype = i
    lib.sgemm_tf32x3_split_a.argtypes = [i, i, vp, i, vp, vp, vp]
    lib.sgemm_tf32x3_split_a.restype = i
    lib.sgemm_tf32x3_split_b.argtypes = [i, i, vp, i, vp, vp, vp]
    lib.sgemm_tf32x3_split_b.restype = i
    lib.sgemm_tf32x3_split_gemm.argtypes = [i, i, i, f, vp, vp, vp, vp, f, vp, i, vp]
    lib.sgemm_tf32x3_split_gemm.restype = i
    lib.sgemm_tf32x3_noalloc.argtypes = gemm
    lib.sgemm_tf32x3_noalloc.restype = i
    lib.reduce_sum_f32.argtypes = [vp, ctypes.c_longlong, vp, vp]
    lib.reduce_sum_f32.restype = i
    lib.sgemm_status_string.argtypes = [i]
    lib.sgemm_status_string.restype = ctypes.c_char_p
    lib.sgemm_last_cuda_error.argtypes = []
    lib.sgemm_last_cuda_error.restype = i
    lib.sgemm_plan_for.argtypes = [i, i, i, f, vp, i, vp, i, f, vp, i, i, i, ctypes.POINTER(Plan)]
    lib.sgemm_plan_for.restype = i
    lib.sgemm_device_status.argtypes = [ctypes.POINTER(i), i]
    lib.sgemm_device_status.restype = i
    lib.sgemm_selftest_wait.argtypes = [ctypes.c_ulonglong, ctypes.POINTER(i)]
    lib.sgemm_selftest_wait.restype = i
    lib.sgemm_bounds_line.argtypes = [ctypes.POINTER(i), i]
    lib.sgemm_bounds_line.restype = i
    lib.sgemm_selftest_bounds.argtypes = [ctypes.POINTER(i)]
    lib.sgemm_selftest_bounds.restype = i
    lib.sgemm_version.argtypes = []
    lib.sgemm_version.restype = ctypes.c_char_p
    return lib


def load(build_if_missing: bool = True, checked: bool = False):
    """The loaded library (ctypes.CDLL): the release one, or with
    checked=True the bounds-checking one.  Raises SgemmError when it is not
    built and cannot be built -- there is no fallback implementation."""
    with _lock:
        if checked not in _libs:
            path = lib_path(checked)
            if build_if_missing:
                path = build(checked=checked)
            if not os.path.exists(path):
                raise SgemmError(-1, f"CUDA library not built ({path}); run __graft_entry__.build()")
            _libs[checked] = _declare(ctypes.CDLL(path))
        return _libs[checked]
