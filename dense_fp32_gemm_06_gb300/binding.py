"""Python binding of the C ABI (argument marshalling only).

Every step of the GEMM runs in the CUDA library; this module turns torch
CUDA tensors (or raw device pointers) into the C call's pointers, leading
dimensions and stream, and turns a non-zero status into ``SgemmError``.
"""
from __future__ import annotations

import ctypes

from . import _native
from ._native import SgemmError

PATH_AUTO = 0
PATH_FFMA = 1
PATH_TF32X3 = 2


def status_string(status: int) -> str:
    return _native.load().sgemm_status_string(int(status)).decode()


def _check(status: int):
    if status:
        lib = _native.load()
        msg = lib.sgemm_status_string(status).decode()
        if status == 100:
            msg += f" (cudaError {lib.sgemm_last_cuda_error()})"
        raise SgemmError(status, msg)


def sgemm_raw(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, stream=0,
              path=PATH_AUTO) -> int:
    """Direct C call on raw device pointers (ints); returns the status."""
    lib = _native.load()
    return lib.sgemm_ex(int(m), int(n), int(k), ctypes.c_float(alpha), ctypes.c_void_p(A_ptr or None),
                        int(lda), ctypes.c_void_p(B_ptr or None), int(ldb), ctypes.c_float(beta),
                        ctypes.c_void_p(C_ptr or None), int(ldc), ctypes.c_void_p(stream or None),
                        int(path))


def plan(m, n, k, alpha=1.0, A_ptr=16, lda=None, B_ptr=16, ldb=None, beta=0.0, C_ptr=16, ldc=None,
         path=PATH_AUTO, num_sms=0):
    """The launch plan the library would use; returns (status, dict).
    num_sms=0 (default): the plan a call on the current device would use (its
    SM count and measured cluster capacity); num_sms > 0: host only (no GPU
    needed) for a device with that many SMs."""
    lib = _native.load()
    lda = max(1, k) if lda is None else lda
    ldb = max(1, n) if ldb is None else ldb
    ldc = max(1, n) if ldc is None else ldc
    p = _native.Plan()
    st = lib.sgemm_plan_for(int(m), int(n), int(k), ctypes.c_float(alpha), ctypes.c_void_p(A_ptr or None),
                            int(lda), ctypes.c_void_p(B_ptr or None), int(ldb), ctypes.c_float(beta),
                            ctypes.c_void_p(C_ptr or None), int(ldc), int(path), int(num_sms),
                            ctypes.byref(p))
    return st, {name: getattr(p, name) for name, _ in _native.Plan._fields_}


def _row_major(t, name):
    import torch
    if t.dtype != torch.float32 or not t.is_cuda or t.dim() != 2:
        raise SgemmError(-1, f"{name} must be a 2-D float32 CUDA tensor")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise SgemmError(-1, f"{name} must have unit column stride (row-major)")
    return max(t.stride(0), 1) if t.shape[0] > 1 else max(t.shape[1], 1)


def sgemm_ex(A, B, C, alpha=1.0, beta=0.0, *, path=PATH_AUTO, stream=None):
    """C = alpha * A @ B + beta * C in place on row-major float32 CUDA tensors
    (A: m x k, B: k x n, C: m x n; any row strides).  Runs on ``stream``
    (default: torch's current stream of C's device).  Returns C."""
    import torch
    m, k = A.shape
    k2, n = B.shape
    if k2 != k or tuple(C.shape) != (m, n):
        raise SgemmError(-1, f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    lda, ldb, ldc = _row_major(A, "A"), _row_major(B, "B"), _row_major(C, "C")
    lda, ldb, ldc = max(lda, k, 1), max(ldb, n, 1), max(ldc, n, 1)
    if stream is None:
        stream = torch.cuda.current_stream(C.device).cuda_stream
    with torch.cuda.device(C.device):
        _check(sgemm_raw(m, n, k, alpha, A.data_ptr(), lda, B.data_ptr(), ldb, beta, C.data_ptr(), ldc,
                         stream, path))
    return C


def sgemm(A, B, C, alpha=1.0, beta=0.0, *, stream=None):
    """C = alpha * A @ B + beta * C (the library's own kernel choice)."""
    return sgemm_ex(A, B, C, alpha, beta, path=PATH_AUTO, stream=stream)


def ka_of(k: int) -> int:
    """Row pitch (floats) of the 3xTF32 split operands: k rounded up to 4."""
    return (int(k) + 3) & ~3


def tf32x3_split_a(A, a_hi, a_lo, *, stream=None):
    """Splits row-major A (m x k) into TF32 hi/lo parts, each m x ka."""
    import torch
    m, k = A.shape
    lda = _row_major(A, "A")
    lda = max(lda, k, 1)
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    with torch.cuda.device(A.device):
        _check(_native.load().sgemm_tf32x3_split_a(m, k, ctypes.c_void_p(A.data_ptr()), lda,
                                                   ctypes.c_void_p(a_hi.data_ptr()),
                                                   ctypes.c_void_p(a_lo.data_ptr()), ctypes.c_void_p(stream or None)))


def tf32x3_split_b(B, bt_hi, bt_lo, *, stream=None):
    """Splits row-major B (k x n) into TF32 hi/lo parts of B^T, each n x ka."""
    import torch
    k, n = B.shape
    ldb = max(_row_major(B, "B"), n, 1)
    if stream is None:
        stream = torch.cuda.current_stream(B.device).cuda_stream
    with torch.cuda.device(B.device):
        _check(_native.load().sgemm_tf32x3_split_b(k, n, ctypes.c_void_p(B.data_ptr()), ldb,
                                                   ctypes.c_void_p(bt_hi.data_ptr()),
                                                   ctypes.c_void_p(bt_lo.data_ptr()), ctypes.c_void_p(stream or None)))


def tf32x3_split_gemm_raw(m, n, k, alpha, a_hi, a_lo, bt_hi, bt_lo, beta, C_ptr, ldc, stream=0) -> int:
    """C = alpha * A @ B + beta * C from split operands (raw device pointers);
    returns the status."""
    return _native.load().sgemm_tf32x3_split_gemm(
        int(m), int(n), int(k), ctypes.c_float(alpha), ctypes.c_void_p(a_hi or None),
        ctypes.c_void_p(a_lo or None), ctypes.c_void_p(bt_hi or None), ctypes.c_void_p(bt_lo or None),
        ctypes.c_float(beta), ctypes.c_void_p(C_ptr or None), int(ldc), ctypes.c_void_p(stream or None))


NOALLOC_SCRATCH_FLOATS = 16 * 1024 * 1024


def tf32x3_noalloc_raw(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, stream=0) -> int:
    """The tensor-core sgemm that allocates no memory (its scratch is a fixed
    64 MiB device array shared by every call); returns the status.  For
    callers that must not allocate device memory while they run; calls that
    overlap on the GPU race on the shared scratch."""
    return _native.load().sgemm_tf32x3_noalloc(
        int(m), int(n), int(k), ctypes.c_float(alpha), ctypes.c_void_p(A_ptr or None), int(lda),
        ctypes.c_void_p(B_ptr or None), int(ldb), ctypes.c_float(beta), ctypes.c_void_p(C_ptr or None), int(ldc),
        ctypes.c_void_p(stream or None))


OP_N = 0
OP_T = 1


def sgemm_op_raw(op_a, op_b, m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, stream=0,
                 path=PATH_AUTO) -> int:
    """C = alpha * op(A) @ op(B) + beta * C on raw device pointers (op_a /
    op_b = OP_N or OP_T, every matrix row-major); returns the status."""
    return _native.load().sgemm_op(
        int(op_a), int(op_b), int(m), int(n), int(k), ctypes.c_float(alpha), ctypes.c_void_p(A_ptr or None),
        int(lda), ctypes.c_void_p(B_ptr or None), int(ldb), ctypes.c_float(beta), ctypes.c_void_p(C_ptr or None),
        int(ldc), ctypes.c_void_p(stream or None), int(path))


def _as_op(t, name):
    """(op, ld) for a 2-D float32 CUDA tensor: a row-major tensor is used as
    is (OP_N), a transposed view of a row-major tensor (unit stride on the
    first axis) reads the underlying matrix transposed (OP_T)."""
    import torch
    if t.dtype != torch.float32 or not t.is_cuda or t.dim() != 2:
        raise SgemmError(-1, f"{name} must be a 2-D float32 CUDA tensor")
    rows, cols = t.shape
    if cols <= 1 or t.stride(1) == 1:
        return OP_N, max(t.stride(0) if rows > 1 else cols, cols, 1)
    if rows <= 1 or t.stride(0) == 1:
        return OP_T, max(t.stride(1) if cols > 1 else rows, rows, 1)
    raise SgemmError(-1, f"{name} must be row-major or a transposed view of a row-major tensor")


def matmul(A, B, C, alpha=1.0, beta=0.0, *, path=PATH_AUTO, stream=None):
    """C = alpha * A @ B + beta * C, where A and B may each be row-major or a
    transposed view (``X.t()``) of a row-major tensor; C must be row-major."""
    import torch
    m, k = A.shape
    k2, n = B.shape
    if k2 != k or tuple(C.shape) != (m, n):
        raise SgemmError(-1, f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    op_a, lda = _as_op(A, "A")
    op_b, ldb = _as_op(B, "B")
    ldc = max(_row_major(C, "C"), n, 1)
    if stream is None:
        stream = torch.cuda.current_stream(C.device).cuda_stream
    with torch.cuda.device(C.device):
        _check(sgemm_op_raw(op_a, op_b, m, n, k, alpha, A.data_ptr(), lda, B.data_ptr(), ldb, beta, C.data_ptr(),
                            ldc, stream, path))
    return C


def sgemm_strided_batched_raw(op_a, op_b, m, n, k, alpha, A_ptr, lda, stride_a, B_ptr, ldb, stride_b, beta, C_ptr,
                              ldc, stride_c, batch, stream=0, path=PATH_AUTO) -> int:
    """`batch` problems C_b = alpha * op(A_b) @ op(B_b) + beta * C_b with
    A_b = A + b*stride_a (floats), and so on; returns the status."""
    return _native.load().sgemm_strided_batched(
        int(op_a), int(op_b), int(m), int(n), int(k), ctypes.c_float(alpha), ctypes.c_void_p(A_ptr or None),
        int(lda), int(stride_a), ctypes.c_void_p(B_ptr or None), int(ldb), int(stride_b), ctypes.c_float(beta),
        ctypes.c_void_p(C_ptr or None), int(ldc), int(stride_c), int(batch), ctypes.c_void_p(stream or None),
        int(path))


def bmm(A, B, C, alpha=1.0, beta=0.0, *, path=PATH_AUTO, stream=None):
    """C[b] = alpha * A[b] @ B[b] + beta * C[b] for 3-D float32 CUDA tensors
    whose last two axes are row-major (or, for A and B, transposed views of
    row-major matrices) and whose first axis has a constant stride (0
    broadcasts one matrix over the batch)."""
    import torch
    if A.dim() != 3 or B.dim() != 3 or C.dim() != 3:
        raise SgemmError(-1, "bmm takes 3-D tensors")
    batch, m, k = A.shape
    _, k2, n = B.shape
    if k2 != k or tuple(C.shape) != (batch, m, n) or B.shape[0] != batch:
        raise SgemmError(-1, f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    op_a, lda = _as_op(A[0], "A")
    op_b, ldb = _as_op(B[0], "B")
    ldc = max(_row_major(C[0], "C"), n, 1)
    if stream is None:
        stream = torch.cuda.current_stream(C.device).cuda_stream
    with torch.cuda.device(C.device):
        _check(sgemm_strided_batched_raw(op_a, op_b, m, n, k, alpha, A.data_ptr(), lda, A.stride(0), B.data_ptr(),
                                         ldb, B.stride(0), beta, C.data_ptr(), ldc, C.stride(0), batch, stream, path))
    return C


def reduce_sum_raw(x_ptr, n, out_ptr, stream=0) -> int:
    """*out = sum of the n floats at x (device pointers); returns the status."""
    return _native.load().reduce_sum_f32(ctypes.c_void_p(x_ptr or None), int(n), ctypes.c_void_p(out_ptr or None),
                                         ctypes.c_void_p(stream or None))


def reduce_sum(x, out=None, *, stream=None):
    """Sum of a contiguous float32 CUDA tensor, as a 1-element tensor."""
    import torch
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise SgemmError(-1, "x must be a contiguous float32 CUDA tensor")
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    with torch.cuda.device(x.device):
        _check(reduce_sum_raw(x.data_ptr(), x.numel(), out.data_ptr(), stream))
    return out


def last_cuda_error() -> int:
    """The CUDA error code behind the calling thread's last status 100."""
    return int(_native.load().sgemm_last_cuda_error())


def device_status(clear: bool = False) -> int:
    """The device-side status word of the tensor-core path (0: no bounded
    wait has run out); synchronises the device; resets it when `clear`."""
    flag = ctypes.c_int(0)
    _check(_native.load().sgemm_device_status(ctypes.byref(flag), int(bool(clear))))
    return flag.value


def selftest_wait_raw(limit_ns: int, gave_up=None) -> int:
    """sgemm_selftest_wait: one bounded wait on a barrier nothing signals;
    returns the status (`gave_up`, a ctypes.c_int, receives the outcome)."""
    return _native.load().sgemm_selftest_wait(ctypes.c_ulonglong(int(limit_ns)),
                                              ctypes.byref(gave_up) if gave_up is not None else None)


def selftest_wait(limit_ns: int = 1_000_000) -> bool:
    """Runs the bounded-wait self-test; True when the wait ran out (it
    should: nothing signals its barrier)."""
    flag = ctypes.c_int(0)
    _check(selftest_wait_raw(limit_ns, flag))
    return flag.value == 1
