"""C-ABI checks that need no GPU: the library builds and loads, exports every
function the header declares, validates arguments with the documented
status codes, and plans launches whose tile bookkeeping agrees with the
two-level blocking model."""
import ctypes
import os
import re

import pytest

import oracle
from dense_fp32_gemm_06_gb300 import _native, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sgemm_gb300.h")


def hplan(*args, **kw):
    """Host-only launch plan for a device with 152 SMs (GB300's count): reads
    no memory and needs no GPU."""
    kw.setdefault("num_sms", 152)
    return binding.plan(*args, **kw)


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:int|const\s+char\s*\*)\s*(\w+)\s*\(", text, flags=re.M)


def test_header_declares_expected_functions():
    names = header_functions()
    assert set(names) == set(_native.EXPORTS), names


def test_library_loads_and_exports_every_symbol():
    lib = _native.load()
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_checked_library_exports_every_symbol():
    """The bounds-checking build (SGEMM_GB300_CHECKED) exports the same C ABI
    and says so in its version string; the release build's bounds self-test
    is refused (status 99) before any CUDA call."""
    lib = _native.load(checked=True)
    for name in header_functions():
        assert hasattr(lib, name), name
    assert lib.sgemm_version().endswith(b"checked)")
    line = ctypes.c_int(-1)
    assert _native.load().sgemm_selftest_bounds(ctypes.byref(line)) == 99
    assert line.value == -1
    assert not _native.load().sgemm_version().endswith(b"checked)")


def test_version_and_status_strings():
    lib = _native.load()
    assert b"sm_103a" in lib.sgemm_version()
    for st in (0, 97, 98, 99, 100):
        s = binding.status_string(st)
        assert s and s != "unknown status"
    # argument errors name the position only: the entry points number their
    # arguments differently (sgemm_op's A is 7, sgemm_strided_batched's C 14)
    for st in range(1, 18):
        assert binding.status_string(st).startswith(f"invalid argument {st} ")
    assert binding.status_string(12345) == "unknown status"


VALID = dict(m=4, n=5, k=6, alpha=1.0, A=256, lda=6, B=512, ldb=5, beta=0.0, C=1024, ldc=5)


def call(**over):
    a = dict(VALID)
    a.update(over)
    # Every case below is rejected (or is a no-op) before any CUDA call, so
    # the fake pointers are never dereferenced.
    return binding.sgemm_raw(a["m"], a["n"], a["k"], a["alpha"], a["A"], a["lda"], a["B"], a["ldb"],
                             a["beta"], a["C"], a["ldc"], 0, a.get("path", 0))


@pytest.mark.parametrize("over,status", [
    (dict(m=-1), 1), (dict(n=-1), 2), (dict(k=-1), 3),
    (dict(A=0), 5), (dict(A=258), 5), (dict(lda=5), 6), (dict(B=0), 7), (dict(B=514), 7),
    (dict(ldb=4), 8), (dict(C=0), 10), (dict(C=1026), 10), (dict(ldc=4), 11),
    (dict(k=0, lda=0), 6), (dict(n=0, ldb=0), 8),
    (dict(m=-1, n=-1), 1), (dict(lda=1, ldc=1), 6),
    (dict(path=7), 98),
])
def test_invalid_arguments(over, status):
    assert call(**over) == status


@pytest.mark.parametrize("over", [dict(m=0), dict(n=0), dict(m=0, A=0, B=0, C=0), dict(n=0, C=0, B=0)])
def test_empty_output_is_a_noop(over):
    assert call(**over) == 0


def test_null_operands_allowed_when_unused():
    # alpha == 0 or k == 0: A and B are not read; plan only (no launch)
    st, p = hplan(4, 5, 6, alpha=0.0, A_ptr=0, B_ptr=0)
    assert st == 0 and p["kernel"] == 1
    st, p = hplan(4, 5, 0, A_ptr=0, B_ptr=0, lda=1)
    assert st == 0 and p["kernel"] == 1


def test_plan_matches_blocking_model():
    """The FFMA plan's grid, threads and slab count at 2048^3 are the
    two-level blocking's M*N blocks, X*Y threads and K big iterations for
    the plan's own tile (bm, bn, bk, rm, rn)."""
    st, p = hplan(2048, 2048, 2048, path=binding.PATH_FFMA)
    assert st == 0
    c = oracle.tiling_counts(2048, 2048, 2048, p["bm"], p["bn"], p["bk"], p["rm"], p["rn"])
    assert p["grid"] == p["tiles"] == c["blocks"]
    assert p["threads"] == c["threads_per_block"]
    assert p["k_tiles"] == c["big_iterations"]
    assert p["smem_bytes"] <= 227 * 1024


def test_ffma_tile_choice(monkeypatch):
    """The FFMA path runs 128 x 128 tiles at two CTAs per SM: 8 x 16 outputs
    per thread (128 threads) from one wave of them on the device's SMs, 8 x 8
    (256 threads) below it; SGEMM_GB300_FFMA_RN pins the per-thread tile."""
    monkeypatch.delenv("SGEMM_GB300_FFMA_RN", raising=False)
    F = binding.PATH_FFMA

    def tile(m, n, k):
        st, p = hplan(m, n, k, path=F)
        assert st == 0
        return p["bm"], p["bn"], p["rm"], p["rn"], p["threads"]

    assert tile(8192, 8192, 8192) == (128, 128, 8, 16, 128)   # 4096 tiles
    assert tile(2432, 2048, 64) == (128, 128, 8, 16, 128)     # 19 x 16 = 304 tiles = 2 x 152
    assert tile(2048, 2048, 2048) == (128, 128, 8, 8, 256)    # 256 tiles
    assert tile(64, 64, 64) == (128, 128, 8, 8, 256)
    monkeypatch.setenv("SGEMM_GB300_FFMA_RN", "16")
    assert tile(64, 64, 64) == (128, 128, 8, 16, 128)
    monkeypatch.setenv("SGEMM_GB300_FFMA_RN", "8")
    assert tile(8192, 8192, 8192) == (128, 128, 8, 8, 256)


def test_plan_ragged_shapes_cover_the_output():
    for m, n, k in ((1000, 1500, 777), (1, 1, 1), (129, 257, 17), (16384, 128, 8192)):
        st, p = hplan(m, n, k, lda=k, path=binding.PATH_FFMA)
        assert st == 0
        assert p["tiles"] == -(-m // p["bm"]) * -(-n // p["bn"])
        assert p["grid"] >= 1 and p["k_tiles"] == -(-k // p["bk"])


def test_plan_alignment_flags():
    st, p = hplan(64, 64, 64, B_ptr=16, C_ptr=16)
    assert (p["b_vec"], p["c_vec"]) == (1, 1)
    st, p = hplan(64, 64, 64, B_ptr=20, C_ptr=16)
    assert (p["b_vec"], p["c_vec"]) == (0, 1)
    st, p = hplan(64, 66, 64, ldb=66, ldc=66)
    assert (p["b_vec"], p["c_vec"]) == (0, 0)


def _split_a(**over):
    a = dict(m=4, k=6, A=256, lda=6, hi=512, lo=1024)
    a.update(over)
    lib = _native.load()
    return lib.sgemm_tf32x3_split_a(a["m"], a["k"], a["A"] or None, a["lda"], a["hi"] or None, a["lo"] or None, None)


def _split_b(**over):
    a = dict(k=6, n=5, B=256, ldb=5, hi=512, lo=1024)
    a.update(over)
    lib = _native.load()
    return lib.sgemm_tf32x3_split_b(a["k"], a["n"], a["B"] or None, a["ldb"], a["hi"] or None, a["lo"] or None, None)


def _split_gemm(**over):
    a = dict(m=4, n=5, k=6, alpha=1.0, ah=256, al=512, bh=768, bl=1024, beta=0.0, C=2048, ldc=5)
    a.update(over)
    return binding.tf32x3_split_gemm_raw(a["m"], a["n"], a["k"], a["alpha"], a["ah"], a["al"], a["bh"], a["bl"],
                                         a["beta"], a["C"], a["ldc"], 0)


@pytest.mark.parametrize("fn,over,status", [
    (_split_a, dict(m=-1), 1), (_split_a, dict(k=-1), 2), (_split_a, dict(A=0), 3), (_split_a, dict(A=258), 3),
    (_split_a, dict(lda=5), 4), (_split_a, dict(hi=0), 5), (_split_a, dict(hi=520), 5), (_split_a, dict(lo=1028), 6),
    (_split_a, dict(m=0, A=0, hi=0, lo=0), 0), (_split_a, dict(k=0, lda=1, A=0, hi=0, lo=0), 0),
    (_split_b, dict(k=-1), 1), (_split_b, dict(n=-1), 2), (_split_b, dict(B=0), 3), (_split_b, dict(ldb=4), 4),
    (_split_b, dict(hi=8), 5), (_split_b, dict(lo=0), 6), (_split_b, dict(n=0, ldb=1, B=0, hi=0, lo=0), 0),
    (_split_gemm, dict(m=-1), 1), (_split_gemm, dict(n=-1), 2), (_split_gemm, dict(k=-1), 3),
    (_split_gemm, dict(ah=0), 5), (_split_gemm, dict(al=520), 6), (_split_gemm, dict(bh=8), 7),
    (_split_gemm, dict(bl=0), 8), (_split_gemm, dict(C=0), 10), (_split_gemm, dict(C=2050), 10),
    (_split_gemm, dict(ldc=4), 11), (_split_gemm, dict(m=0, ah=0, al=0, bh=0, bl=0, C=0), 0),
])
def test_split_api_arguments(fn, over, status):
    # every case is rejected, or is a no-op, before any CUDA call
    assert fn(**over) == status


def test_auto_policy():
    """AUTO takes the tensor-core path from 2^20 multiply-adds with k >= 64,
    or for k > 8192; the FFMA path for smaller problems and shorter k."""
    assert hplan(64, 64, 64)[1]["path"] == binding.PATH_FFMA
    assert hplan(100, 100, 100)[1]["path"] == binding.PATH_FFMA       # 10^6 < 2^20
    assert hplan(128, 128, 64)[1]["path"] == binding.PATH_TF32X3      # 2^20
    assert hplan(256, 256, 256)[1]["path"] == binding.PATH_TF32X3
    assert hplan(4096, 4096, 32)[1]["path"] == binding.PATH_FFMA     # k < 64
    assert hplan(4096, 4096, 63)[1]["path"] == binding.PATH_FFMA
    assert hplan(4096, 4096, 64)[1]["path"] == binding.PATH_TF32X3
    assert hplan(512, 512, 512)[1]["path"] == binding.PATH_TF32X3
    assert hplan(8192, 8192, 8192)[1]["path"] == binding.PATH_TF32X3
    assert hplan(16, 16, 8193)[1]["path"] == binding.PATH_TF32X3
    assert hplan(1000, 1500, 777, lda=777)[1]["path"] == binding.PATH_TF32X3
    st, p = hplan(2048, 2048, 2048, path=binding.PATH_TF32X3)     # CTA pairs: 8 x 8 tiles of 256 x 256
    assert st == 0 and (p["bm"], p["bn"], p["bk"], p["threads"], p["pair"]) == (256, 256, 16, 384, 1)
    assert p["tiles"] == 8 * 8 and p["grid"] == 2 * p["tiles"] and p["k_tiles"] == 128 and p["stream_k"] == 0
    st, p = hplan(8192, 8192, 8192, path=binding.PATH_TF32X3)     # many waves: single CTAs, stream-K
    assert st == 0 and (p["bm"], p["bn"], p["pair"]) == (128, 256, 0) and p["tiles"] == 64 * 32
    assert p["stream_k"] == 152 and p["grid"] == 152 and p["persistent"] == 0


def test_persistent_policy(monkeypatch):
    """Whole tiles of more than one wave run on one persistent CTA per SM
    (tiles g, g + 152, ...); not for split-K, stream-K, CTA pairs or
    batches, nor within one wave; SGEMM_GB300_PERSIST pins it off."""
    for v in ("SGEMM_GB300_PERSIST", "SGEMM_GB300_STREAM_K", "SGEMM_GB300_PAIR"):
        monkeypatch.delenv(v, raising=False)
    TC = binding.PATH_TF32X3

    def plan(m, n, k):
        st, p = hplan(m, n, k, path=TC)
        assert st == 0
        return p

    p = plan(8192, 4864, 4096)                 # 64 x 19 = 1216 tiles = 8 waves exactly
    assert p["persistent"] == 1 and p["grid"] == 152 and p["tiles"] == 1216 and p["stream_k"] == 0
    p = plan(3000, 2600, 300)                  # 264 tiles: stream-K's fix-up would cost more
    assert p["persistent"] == 1 and p["stream_k"] == 0
    p = plan(2176, 2304, 512)                  # 17 x 9 = 153 tiles: one more than a wave
    assert (p["tiles"], p["persistent"], p["grid"]) == (153, 1, 152)
    monkeypatch.setenv("SGEMM_GB300_PAIR", "0")
    p = plan(2048, 2304, 512)                  # 16 x 9 = 144 tiles: one wave
    assert p["tiles"] == 144 and p["persistent"] == 0 and p["grid"] == p["tiles"] * p["split_k"]
    monkeypatch.delenv("SGEMM_GB300_PAIR")
    assert plan(4096, 4096, 4096)["persistent"] == 0          # stream-K
    assert plan(2048, 2048, 2048)["persistent"] == 0          # CTA pairs
    monkeypatch.setenv("SGEMM_GB300_PERSIST", "0")
    p = plan(8192, 4864, 4096)
    assert p["persistent"] == 0 and p["grid"] == p["tiles"] == 1216


def test_stream_k_policy(monkeypatch):
    """Stream-K (one CTA per SM: the full waves as whole tiles, the last
    wave's tiles shared out by slabs) when its estimate beats whole tiles and
    split-K; never for batches, never when a tile would meet too many CTAs
    (few tiles: split-K clusters instead), never with fewer slabs than CTAs;
    the tuning variable pins it."""
    for v in ("SGEMM_GB300_STREAM_K", "SGEMM_GB300_TRANS", "SGEMM_GB300_TILE_N", "SGEMM_GB300_SPLIT_K"):
        monkeypatch.delenv(v, raising=False)
    TC = binding.PATH_TF32X3
    for shape in [(4096, 4096, 4096), (8192, 2048, 8192), (16384, 128, 8192), (65536, 64, 4096), (8192, 8192, 8192)]:
        st, p = hplan(*shape, path=TC)
        assert st == 0 and p["stream_k"] == 152 and p["grid"] == 152 and p["split_k"] == 1, (shape, p)
    # 2048^3: CTA pairs; 3072^3: the estimate ties; 8192 x 4864: whole waves
    for shape in [(2048, 2048, 2048), (3072, 3072, 3072), (8192, 4864, 4096)]:
        st, p = hplan(*shape, path=TC)
        expect = 152 if p["persistent"] else p["tiles"] * p["split_k"] * (2 if p["pair"] else 1)
        assert p["stream_k"] == 0 and p["grid"] == expect, (shape, p)
    st, p = hplan(256, 256, 8192, path=TC)          # 2 tiles: a split-K cluster instead
    assert p["stream_k"] == 0 and p["split_k"] > 1
    st, p = hplan(4096, 4096, 4096, path=TC, num_sms=64)
    assert p["stream_k"] == 0 and p["tiles"] == 512 and p["grid"] == 64   # 8 full waves of 64: persistent
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "0")
    st, p = hplan(4096, 4096, 4096, path=TC)
    assert p["stream_k"] == 0 and p["persistent"] == 1 and p["grid"] == 152
    monkeypatch.setenv("SGEMM_GB300_STREAM_K", "1")
    for shape in [(256, 256, 8192), (2048, 2048, 2048)]:    # pinned: taken whenever allowed
        st, p = hplan(*shape, path=TC)
        assert p["stream_k"] == 152 and p["grid"] == 152, (shape, p)
    st, p = hplan(64, 64, 32, path=TC)               # 1 tile x 2 slabs < 152 CTAs
    assert p["stream_k"] == 0


def test_stream_k_parts_policy(monkeypatch):
    """After two or more full waves, a stream-K plan cuts each of the R tiles
    left into S = sms / R equal k parts, one per CTA (when S >= 2); with no
    full wave, or S = 1, the slab sequence is cut into equal runs.
    SGEMM_GB300_SK_PARTS pins the choice."""
    for v in ("SGEMM_GB300_STREAM_K", "SGEMM_GB300_TRANS", "SGEMM_GB300_TILE_N", "SGEMM_GB300_SPLIT_K",
              "SGEMM_GB300_SK_PARTS"):
        monkeypatch.delenv(v, raising=False)
    TC = binding.PATH_TF32X3
    # 8192^3: 2048 tiles = 13 x 152 + 72 -> 2 parts; 4096^3: 512 = 3 x 152 + 56 -> 2
    for shape, S in [((8192, 8192, 8192), 2), ((4096, 4096, 4096), 2), ((8192, 2048, 8192), 2),
                     ((16384, 128, 8192), 0), ((6144, 6144, 6144), 0)]:
        st, p = hplan(*shape, path=TC)
        assert st == 0 and p["stream_k"] == 152 and p["sk_parts"] == S, (shape, p)
    monkeypatch.setenv("SGEMM_GB300_SK_PARTS", "0")
    st, p = hplan(8192, 8192, 8192, path=TC)
    assert p["stream_k"] == 152 and p["sk_parts"] == 0
    monkeypatch.setenv("SGEMM_GB300_SK_PARTS", "1")
    st, p = hplan(16384, 128, 8192, path=TC)        # pinned: 64 tiles, 2 parts each
    assert p["stream_k"] == 152 and p["sk_parts"] == 2
    st, p = hplan(2048, 2048, 2048, path=TC)        # CTA pairs: no stream-K, no parts
    assert p["stream_k"] == 0 and p["sk_parts"] == 0


def test_raster_group_policy(monkeypatch):
    """Raster groups of 24 tile rows where the operands as read (4 bytes a
    value as stored, 8 split) exceed twice L2, of 8 otherwise (capped at the
    tile rows); SGEMM_GB300_GROUP_M pins it."""
    monkeypatch.delenv("SGEMM_GB300_GROUP_M", raising=False)
    TC = binding.PATH_TF32X3
    for shape, g in [((8192, 8192, 8192), 24), ((8192, 8192, 4096), 24), ((16384, 8192, 4096), 24),
                     ((4096, 4096, 4096), 8), ((1000, 1500, 777), 8), ((256, 256, 256), 2)]:
        st, p = hplan(*shape, path=TC)
        assert st == 0 and p["group_m"] == g, (shape, p)
    monkeypatch.setenv("SGEMM_GB300_GROUP_M", "12")
    st, p = hplan(8192, 8192, 8192, path=TC)
    assert p["group_m"] == 12


def test_in_kernel_split_policy(monkeypatch):
    """The tensor-core GEMM reads an operand as stored and splits it itself
    when TMA can load it -- a 16-byte aligned base, rows a multiple of 16
    bytes and, in a batch, a stride of 0 or of whole non-overlapping matrices
    16 bytes apart; otherwise a split pass writes that operand's hi and lo
    parts into scratch -- except an A that TMA cannot read on untransposed
    single-CTA tiles, which the GEMM reads in four row phases.  A is
    read as stored whenever it can be; B (whose split costs the GEMM more per
    slab) for m*n*k <= 2^31, and above that on CTA pairs when their 256 x 256
    tiles fill 3/4 to all of the pair slots in one wave.  The tuning variables
    pin the choice but cannot make an unaligned B eligible.  Every
    tensor-core plan runs 12 warps."""
    for v in ("SGEMM_GB300_SPLIT_A_IN", "SGEMM_GB300_SPLIT_B_IN"):
        monkeypatch.delenv(v, raising=False)
    TC = binding.PATH_TF32X3

    def raw(m, n, k, **kw):
        st, p = hplan(m, n, k, path=TC, **kw)
        assert st == 0
        assert p["threads"] == 384
        return p["a_in_kernel"], p["b_in_kernel"]

    assert raw(16384, 128, 8192) == (1, 0)
    assert raw(8192, 8192, 8192) == (1, 0)
    assert raw(2048, 2048, 2048) == (1, 1)                # one wave of CTA pairs, which read B as stored
    assert raw(2048, 2048, 2048, B_ptr=24) == (1, 0)      # B not 16-byte aligned: single CTAs, B split first
    assert raw(3072, 2048, 2048) == (1, 0)                # 96 pair tiles: more than one wave
    assert raw(1024, 1024, 2048) == (1, 1)                # 2^31 multiply-adds
    assert raw(1024, 1024, 2049, lda=2052) == (1, 0)      # one k more
    assert raw(256, 256, 256) == (1, 1)
    assert raw(1000, 1500, 777) == (1, 1)                 # lda = 777: A read in row phases
    assert raw(1000, 1500, 777, lda=780) == (1, 1)
    assert raw(1000, 1500, 780, A_ptr=20) == (1, 1)       # A not 16-byte aligned: row phases too
    assert raw(16384, 128, 8191) == (0, 0)                # transposed tiles (A on the n side): A split first
    assert raw(2048, 2048, 2048, lda=2049) == (1, 0)      # phased A: single CTAs, so B split first
    assert raw(1000, 1500, 780, B_ptr=24) == (1, 0)       # B not 16-byte aligned
    assert raw(1000, 1498, 780) == (1, 0)                 # ldb = 1498: B's rows not 16-byte aligned
    monkeypatch.setenv("SGEMM_GB300_SPLIT_B_IN", "1")
    assert raw(16384, 128, 8192) == (1, 1)
    assert raw(1000, 1498, 780) == (1, 0)
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", "0")
    monkeypatch.setenv("SGEMM_GB300_SPLIT_B_IN", "0")
    assert raw(256, 256, 256) == (0, 0)
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", "1")
    monkeypatch.setenv("SGEMM_GB300_SPLIT_B_IN", "1")
    assert raw(8192, 8192, 8192) == (1, 1)
    assert raw(1000, 1500, 777) == (1, 1)
    monkeypatch.setenv("SGEMM_GB300_SPLIT_A_IN", "0")
    assert raw(1000, 1500, 777) == (0, 1)


def test_op_argument_checks():
    """sgemm_op rejects bad ops and leading dimensions before any CUDA call."""
    assert binding.sgemm_op_raw(2, 0, 4, 4, 4, 1.0, 256, 4, 512, 4, 0.0, 1024, 4) == 1
    assert binding.sgemm_op_raw(0, 5, 4, 4, 4, 1.0, 256, 4, 512, 4, 0.0, 1024, 4) == 2
    # op(A) = A^T with A stored k x m: lda must cover m
    assert binding.sgemm_op_raw(1, 0, 8, 4, 4, 1.0, 256, 4, 512, 4, 0.0, 1024, 4) == 8
    # op(B) = B^T with B stored n x k: ldb must cover k
    assert binding.sgemm_op_raw(0, 1, 4, 4, 8, 1.0, 256, 8, 512, 4, 0.0, 1024, 4) == 10


def test_strided_batched_argument_checks():
    """Positions: op_a 1, op_b 2, m 3, n 4, k 5, A 7, lda 8, stride_a 9, B 10,
    ldb 11, stride_b 12, C 14, ldc 15, stride_c 16, batch 17."""
    def call(**o):
        a = dict(op_a=0, op_b=0, m=4, n=5, k=6, A=256, lda=6, sa=24, B=512, ldb=5, sb=30, C=1024, ldc=5, sc=20,
                 batch=3)
        a.update(o)
        return binding.sgemm_strided_batched_raw(a["op_a"], a["op_b"], a["m"], a["n"], a["k"], 1.0, a["A"],
                                                 a["lda"], a["sa"], a["B"], a["ldb"], a["sb"], 0.0, a["C"], a["ldc"],
                                                 a["sc"], a["batch"], 0)
    assert call(op_a=3) == 1 and call(op_b=-1) == 2
    assert call(m=-1) == 3 and call(n=-1) == 4 and call(k=-1) == 5
    assert call(A=0) == 7 and call(lda=5) == 8 and call(sa=-1) == 9
    assert call(B=0) == 10 and call(ldb=4) == 11 and call(sb=-4) == 12
    assert call(C=0) == 14 and call(ldc=4) == 15
    assert call(sc=19) == 16          # C matrices would overlap: (m-1)*ldc + n = 20
    assert call(batch=-1) == 17
    assert call(batch=0) == 0 and call(m=0) == 0


def test_trans_tile_policy(monkeypatch):
    """n <= 128 may take transposed 256 x 128 tiles (C^T = B^T A^T) when the
    plan's estimate favours them; n > 128 never does; the tuning variable
    pins the choice."""
    for v in ("SGEMM_GB300_TRANS", "SGEMM_GB300_TILE_N", "SGEMM_GB300_SPLIT_K"):
        monkeypatch.delenv(v, raising=False)
    TC = binding.PATH_TF32X3
    st, p = hplan(16384, 128, 8192, path=TC)
    assert st == 0 and p["trans"] == 1 and (p["bm"], p["bn"], p["stages"]) == (256, 128, 4)
    assert p["tiles"] == 64 and p["grid"] == (p["stream_k"] or 64 * p["split_k"])
    assert hplan(65536, 64, 4096, path=TC)[1]["trans"] == 1
    assert hplan(8192, 129, 8192, path=TC)[1]["trans"] == 0
    assert hplan(8192, 8192, 8192, path=TC)[1]["trans"] == 0
    monkeypatch.setenv("SGEMM_GB300_TRANS", "0")
    assert hplan(16384, 128, 8192, path=TC)[1]["trans"] == 0
    monkeypatch.setenv("SGEMM_GB300_TRANS", "1")
    st, p = hplan(300, 100, 5000, path=TC)
    assert p["trans"] == 1 and (p["bm"], p["bn"]) == (256, 128)
    assert hplan(300, 200, 5000, path=TC)[1]["trans"] == 0


def test_device_plan_needs_a_device():
    """The default plan is the current device's (num_sms=0); without a usable device
    that is a CUDA error (status 100), reported, not guessed."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    st, _ = binding.plan(2048, 2048, 2048)
    assert st == 100


def test_selftest_wait_argument_checks():
    """The bounded-wait self-test rejects its arguments before any CUDA call."""
    import ctypes
    flag = ctypes.c_int(-1)
    assert binding.selftest_wait_raw(0, flag) == 1                  # no limit
    assert binding.selftest_wait_raw(10_000_000_001, flag) == 1     # over 10 s
    assert binding.selftest_wait_raw(1_000_000, None) == 2          # no result pointer
    assert flag.value == -1


def test_split_k_policy_small_and_large_shapes():
    """Host plan (152 SMs, no device): small problems with few tiles split k
    over clusters (a split costs ~2 us + 0.5 us per CTA and leaves each CTA
    >= 4 slabs); problems that fill the GPU with whole tiles do not."""
    TC = binding.PATH_TF32X3
    expect = {(256, 256, 256): 4, (384, 384, 384): 4, (500, 500, 300): 4, (256, 256, 8192): 8,
              (128, 128, 128): 1, (2048, 2048, 2048): 1, (8192, 8192, 8192): 1}
    for (m, n, k), s in expect.items():
        st, p = hplan(m, n, k, lda=k, path=TC, num_sms=152)
        assert st == 0 and p["split_k"] == s, ((m, n, k), p)
        assert p["grid"] == (152 if p["persistent"] or p["stream_k"] else p["tiles"] * s * (2 if p["pair"] else 1))
        assert p["k_tiles"] // p["split_k"] >= 4 or s == 1
