/*
 * sgemm_gb300.h -- C ABI of a single-precision GEMM for NVIDIA GB300 (sm_103a).
 *
 *     C = alpha * A * B + beta * C        A: m x k, B: k x n, C: m x n, FP32
 *
 * Operation.  C_ij = sum_{t=0}^{k-1} A_it * B_tj is the GEMM definition of
 * hatrix.site "GEMM优化原理" (section 问题定义, first equation; also
 * aerisun.top "GPU 访存与计算优化", section "Naive GEMM 的重复读取").  The pages
 * call the kernel with two float scalars next to the three matrices and the
 * three sizes (blog.lightlisten.com "gemm优化", the ncu launch line in section
 * 实际测试：ncu); they say nothing further about the scalars, so alpha and beta
 * take the BLAS meaning: beta == 0 makes C write-only (its old contents are
 * never read, so NaN there does not propagate), and alpha == 0 or k == 0
 * gives C = beta * C without reading A or B.
 *
 * Layout.  Row-major with leading dimensions, as the pages' loads assume
 * (aerisun.top, section "Shared Tiling 与 block 内复用"):
 *     A(i,t) = A[i*lda + t],  B(t,j) = B[t*ldb + j],  C(i,j) = C[i*ldc + j].
 * Offsets are computed in 64 bits.  Any lda >= max(1,k), ldb >= max(1,n),
 * ldc >= max(1,n) and any 4-byte-aligned pointers are accepted by both
 * paths (the FFMA path copies A 4 bytes at a time and B / C 16 bytes at a
 * time where their rows are 16-byte aligned; the tensor-core path re-lays
 * A and B out itself, see the split calls below).
 *
 * Ownership.  A, B and C are device pointers owned by the caller (any memory
 * the current device can address).  The library keeps no pointer after the
 * call returns.  Per device it lazily caches kernel attributes and its
 * cluster capacity.  The FFMA path allocates nothing.  The tensor-core GEMM
 * reads an operand as stored (by TMA) and splits it into TF32 parts itself
 * when the operand's base is 16-byte aligned and its rows are 16 bytes
 * apart (lda, ldb multiples of 4; in a batch also a stride of 0 or of whole
 * non-overlapping matrices, a multiple of 4) -- always for A, and for B
 * when m*n*k <= 2^31 or the plan runs CTA pairs (other large problems
 * split B with a separate pass, which is faster there).  An A (not
 * transposed) whose rows are not 16 bytes apart, or whose base is not
 * 16-byte aligned, the GEMM reads in four row phases (rows j, j + 4, ...
 * are 4 * lda floats apart, which TMA can read) and needs no scratch for it
 * either, except on transposed tiles (sgemm_plan.trans) and in a batch
 * whose stride is not a multiple of 4.  Only the other operands, and
 * stream-K's partial tiles
 * (plans with sgemm_plan.stream_k > 0), take scratch: 8 * rows * ka bytes
 * per split operand (ka = k rounded up to 4) and 2 * stream_k tiles of
 * 128 * bn floats, for the duration of the call, from a stream-ordered
 * memory pool the library creates per device on first use
 * (cudaMallocFromPoolAsync / cudaFreeAsync on `stream`).  A call that needs
 * no scratch allocates nothing.  The pool keeps up to 2 GiB mapped between
 * calls (environment variable SGEMM_GB300_POOL_KEEP_MB overrides it, read
 * once per device), so repeated calls do not map and unmap device memory;
 * it is released when the process exits.  sgemm_plan_for() tells which
 * case a problem is (a_in_kernel, b_in_kernel, stream_k).  C must not
 * overlap A or B.
 *
 * Execution.  Every entry point that takes a stream enqueues its kernels on
 * `stream` (0 = the legacy default stream) of the current device and returns
 * without synchronising; errors raised later by the GPU surface at the
 * caller's next synchronisation.  Calls are thread-safe, and calls on
 * different streams may run at the same time (each takes its scratch from
 * the pool in its own stream's order).  A call of sgemm, sgemm_ex, sgemm_op
 * or sgemm_strided_batched may be captured into a CUDA graph once an earlier
 * call has done the device's one-time set-up (kernel attributes, the
 * scratch pool): its pool allocation, the counter reset of stream-K and its
 * launches become graph nodes.  The library keeps per-device state from
 * its first call on a device (kernel attributes, cluster capacity, the
 * scratch pool, the device address of the no-allocation scratch); calls
 * made after cudaDeviceReset() on a device it has already used are not
 * supported.
 *
 * Errors.  The return value is a status:
 *     0                      success;
 *     1 .. 11                argument i (1-based, BLAS "info" convention) is
 *                            invalid: 1 m < 0, 2 n < 0, 3 k < 0,
 *                            5 A == NULL while m*n*k > 0 and alpha != 0,
 *                            6 lda < max(1,k), 7 B == NULL (same rule as A),
 *                            8 ldb < max(1,n), 10 C == NULL while m*n > 0,
 *                            11 ldc < max(1,n); also 5/7/10 for a pointer not
 *                            4-byte aligned;
 *     SGEMM_STATUS_TOO_LARGE  sgemm_tf32x3_noalloc(): the problem does not fit
 *                            its fixed scratch array;
 *     SGEMM_STATUS_BAD_PATH  sgemm_ex() asked for an unknown path;
 *     SGEMM_STATUS_UNSUPPORTED  sgemm_plan_for() was given a NULL plan, or
 *                            sgemm_selftest_bounds() ran in a release build;
 *     SGEMM_STATUS_CUDA_ERROR  a CUDA runtime call or launch failed; the CUDA
 *                            error code is kept per thread and returned by
 *                            sgemm_last_cuda_error().
 * Argument errors, a failed scratch allocation and a failed tensor-map
 * encoding return before anything is enqueued.  A launch that fails
 * (status SGEMM_STATUS_CUDA_ERROR from the launch itself) may leave earlier
 * kernels of the same call enqueued; sgemm_strided_batched with more than
 * 65535 problems runs one chunk of 65535 after another and stops at the
 * first chunk that fails.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SGEMM_STATUS_OK 0
#define SGEMM_STATUS_TOO_LARGE 97
#define SGEMM_STATUS_BAD_PATH 98
#define SGEMM_STATUS_UNSUPPORTED 99
#define SGEMM_STATUS_CUDA_ERROR 100

/* Kernel families sgemm_ex() can be asked for. */
#define SGEMM_PATH_AUTO 0   /* the library's choice (what sgemm() runs): TF32X3 when
                               m*n*k >= 2^20 and k >= 64, or k > 8192; else FFMA */
#define SGEMM_PATH_FFMA 1   /* CUDA-core FP32 FFMA, exact FP32 products        */
#define SGEMM_PATH_TF32X3 2 /* tcgen05 tensor cores, 3xTF32 split precision    */

/*
 * sgemm -- C = alpha * A * B + beta * C on `stream`.  See the file comment
 * for layout, ownership and status codes.
 */
int sgemm(int m, int n, int k, float alpha,
          const float *A, int lda, const float *B, int ldb,
          float beta, float *C, int ldc, cudaStream_t stream);

/*
 * sgemm_ex -- as sgemm, with the kernel family chosen by `path`
 * (SGEMM_PATH_*).  SGEMM_PATH_AUTO is identical to sgemm().
 */
int sgemm_ex(int m, int n, int k, float alpha,
             const float *A, int lda, const float *B, int ldb,
             float beta, float *C, int ldc, cudaStream_t stream, int path);

/*
 * sgemm_op -- C = alpha * op(A) * op(B) + beta * C, op(A) m x k, op(B) k x n,
 * every matrix row-major.  The pages define only the untransposed product
 * (hatrix.site "GEMM优化原理", section 问题定义); the transposed forms are the
 * same sum over t with the operands read in the other order:
 *   op_a == SGEMM_OP_N: A stored m x k, op(A)(i,t) = A[i*lda + t], lda >= max(1,k);
 *   op_a == SGEMM_OP_T: A stored k x m, op(A)(i,t) = A[t*lda + i], lda >= max(1,m);
 *   op_b == SGEMM_OP_N: B stored k x n, op(B)(t,j) = B[t*ldb + j], ldb >= max(1,n);
 *   op_b == SGEMM_OP_T: B stored n x k, op(B)(t,j) = B[j*ldb + t], ldb >= max(1,k).
 * (Column-major BLAS data maps onto this by C^T = op(B)^T op(A)^T.)
 * Status positions count op_a as 1 and op_b as 2 (m is 3, ..., ldc 13).
 */
#define SGEMM_OP_N 0
#define SGEMM_OP_T 1
int sgemm_op(int op_a, int op_b, int m, int n, int k, float alpha,
             const float *A, int lda, const float *B, int ldb,
             float beta, float *C, int ldc, cudaStream_t stream, int path);

/*
 * sgemm_strided_batched -- `batch` independent products of one shape,
 *     C_b = alpha * op(A_b) * op(B_b) + beta * C_b,   b = 0 .. batch-1,
 * with A_b = A + b*stride_a, B_b = B + b*stride_b, C_b = C + b*stride_c
 * (strides in floats).  Not on the pages; the same operation per problem.
 * A stride of 0 shares that operand across the batch; the C matrices must
 * not overlap (stride_c >= (m-1)*ldc + n when batch > 1).  Each path runs
 * the whole batch in one launch per kernel (grid y = problem; batches
 * beyond 65535 problems go in chunks).  Status positions: op_a 1, op_b 2,
 * m 3, n 4, k 5, A 7, lda 8, stride_a 9, B 10, ldb 11, stride_b 12, C 14,
 * ldc 15, stride_c 16, batch 17.  batch == 0 is a no-op (the pointers
 * are not looked at).
 */
int sgemm_strided_batched(int op_a, int op_b, int m, int n, int k, float alpha,
                          const float *A, int lda, long long stride_a,
                          const float *B, int ldb, long long stride_b,
                          float beta, float *C, int ldc, long long stride_c,
                          int batch, cudaStream_t stream, int path);


/*
 * 3xTF32 split operands.  The pages describe only CUDA-core FFMA kernels;
 * the tensor-core path computes the same C = alpha*A*B + beta*C by writing
 * each FP32 operand x as two TF32 numbers, hi = tf32(x) and
 * lo = tf32(x - hi) (both rounded to nearest), and summing
 * a_hi*b_hi + a_hi*b_lo + a_lo*b_hi on the tensor cores in 128-deep chunks
 * whose sums are added in FP32 on the CUDA cores.  sgemm_ex(...,
 * SGEMM_PATH_TF32X3) does all of it: an operand TMA can read as stored is
 * split inside the GEMM kernel (hi = x with its low 13 mantissa bits
 * dropped, which is how the tensor core reads an FP32 operand, and
 * lo = tf32(x - hi) rounded to nearest), the others by a split pass into
 * scratch (see Ownership above).  A caller that multiplies the same operand
 * many times can split it once with these calls and reuse it.
 *
 * Split layout: ka = k rounded up to a multiple of 4.  a_hi, a_lo are
 * m x ka row-major (row pitch ka floats); bt_hi, bt_lo hold B TRANSPOSED,
 * n x ka row-major.  Columns k .. ka-1 are never read or written.  Every
 * split array must be 16-byte aligned and hold rows*ka floats; the caller
 * owns them.
 *
 * Status: 0, or the 1-based position of the first invalid argument
 * (sizes < 0; A/B NULL or not 4-byte aligned; lda < max(1,k),
 * ldb < max(1,n); a split array NULL or not 16-byte aligned while there is
 * work), or SGEMM_STATUS_CUDA_ERROR.  Asynchronous on `stream`.
 */
int sgemm_tf32x3_split_a(int m, int k, const float *A, int lda, float *a_hi, float *a_lo, cudaStream_t stream);
int sgemm_tf32x3_split_b(int k, int n, const float *B, int ldb, float *bt_hi, float *bt_lo, cudaStream_t stream);

/*
 * C = alpha * A * B + beta * C from split operands (argument positions as
 * in sgemm: 5..8 are a_hi, a_lo, bt_hi, bt_lo; 10 C; 11 ldc).  Runs only
 * the tensor-core GEMM kernel (k == 0 or alpha == 0: C = beta * C).
 */
int sgemm_tf32x3_split_gemm(int m, int n, int k, float alpha, const float *a_hi, const float *a_lo,
                            const float *bt_hi, const float *bt_lo, float beta, float *C, int ldc,
                            cudaStream_t stream);

/*
 * sgemm_tf32x3_noalloc -- the tensor-core (3xTF32) sgemm with no memory
 * allocation of any kind.  The pages have no counterpart to this entry
 * point; it exists for callers that must not allocate device memory while
 * they run: code executing inside an allocator callback or an out-of-memory
 * handler, processes that reserve all of their device memory up front, and
 * latency-critical loops that cannot afford cudaMalloc / cudaMallocAsync
 * (which can synchronise, fail under memory pressure, or take a lock the
 * caller already holds).
 *
 * Arguments, layout, results and status codes are those of sgemm() with the
 * tensor-core path, plus SGEMM_STATUS_TOO_LARGE.  Every operand whose rows
 * are 16 bytes apart and whose base is 16-byte aligned is read as stored
 * and split inside the GEMM, whatever the problem's size (problems above
 * 2^31 multiply-adds with both operands so run on CTA pairs: 256 x 256
 * tiles, cta_group::2), and an A that is not is read in row phases as in
 * sgemm(), so such calls need no scratch at all.  The split parts of the
 * other operands -- a B whose rows TMA cannot read, and such an A on
 * transposed tiles (sgemm_plan.trans) -- live in one fixed array of
 * SGEMM_NOALLOC_SCRATCH_FLOATS floats (64 MiB) in device memory that every
 * GPU which loads this library holds until the process exits: 2 * rows * ka
 * floats per such operand (rows = m for A, n for B; ka = k rounded up to
 * 4); a problem that needs more is rejected with SGEMM_STATUS_TOO_LARGE
 * before anything is enqueued (with B's rows misaligned, n = 4096 and
 * k = 2048 need exactly the capacity).  No stream-K.  No cudaMalloc,
 * cudaMallocAsync, cudaFree or allocating library routine is called.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with the device current) and keeps it; make
 * that first call before any stream capture is begun.  All calls share the
 * one array and it keeps whatever the last call left there (nothing in it
 * needs to start at zero: every element a call reads was written earlier in
 * the same call).  Two calls whose work overlaps on the GPU -- on different
 * streams, or on different host threads -- race on the array and corrupt
 * each other's results; serialise them (one stream, or events).
 */
#define SGEMM_NOALLOC_SCRATCH_FLOATS (16 * 1024 * 1024)
int sgemm_tf32x3_noalloc(int m, int n, int k, float alpha,
                         const float *A, int lda, const float *B, int ldb,
                         float beta, float *C, int ldc, cudaStream_t stream);

/*
 * reduce_sum_f32 -- *out = sum_{i<n} x[i] (FP32), the block reduction of
 * aerisun.top "GPU 访存与计算优化", section "Reduce 的分层归约": per-thread
 * register sums over a grid-stride loop, warp shuffles, a shared-memory
 * combine per block and one atomic add per block into *out (which the call
 * zeroes first on `stream`).  x and out are device pointers (x 4-byte
 * aligned).
 *
 * Launch shape: B = min(ceil(n / (16 * SGEMM_REDUCE_THREADS)),
 * SGEMM_REDUCE_BLOCKS_PER_SM * SMs) blocks (at least 1) of
 * SGEMM_REDUCE_THREADS threads, G = B * SGEMM_REDUCE_THREADS threads in all.
 * With x 16-byte aligned, thread g reads float4 g, g + G, g + 2G, ... and
 * adds component c of each into accumulator c (four FP32 accumulators),
 * the n % 4 values after the last whole float4 going one each into the
 * first accumulator of threads 0 .. n%4-1; otherwise every value goes
 * through 4-byte loads into the first accumulator.  Then
 * (a0 + a1) + (a2 + a3), a 5-level shuffle tree over the warp, the same
 * tree over the block's warp sums, and the B block sums are added into *out
 * one after another.  The longest chain of additions is therefore
 *     h = ceil(floor(n/4) / G) + (n % 4 != 0) + 12 + B   (x 16-byte aligned)
 *     h = ceil(n / G) + 12 + B                            (otherwise)
 * and the result is within gamma_h * sum|x_i| of the exact sum
 * (gamma_h = h u / (1 - h u), u = 2^-24).  The order in which blocks commit
 * is not fixed, so the last bits of the sum may differ between runs.
 * Status: 1 x NULL / misaligned while n > 0, 2 n < 0, 3 out NULL /
 * misaligned, SGEMM_STATUS_CUDA_ERROR.  n == 0 gives 0.
 */
#define SGEMM_REDUCE_THREADS 512
#define SGEMM_REDUCE_BLOCKS_PER_SM 4
int reduce_sum_f32(const float *x, long long n, float *out, cudaStream_t stream);

/* Static, NUL-terminated description of a status code. */
const char *sgemm_status_string(int status);

/* cudaError_t value of the last SGEMM_STATUS_CUDA_ERROR on this thread. */
int sgemm_last_cuda_error(void);

/*
 * Launch plan the library would use for a problem.  The pointers are
 * inspected for alignment only.  num_sms > 0: host only (reads no memory,
 * needs no GPU) for a device with that many SMs (152 on GB300), assuming
 * clusters of S CTAs fill GPCs of num_sms / 8 SMs.  num_sms == 0: the plan
 * for the current device, with its measured cluster capacity -- the plan a
 * call made now would use (the device's one-time set-up runs if needed).
 */
typedef struct sgemm_plan {
    int path;          /* SGEMM_PATH_FFMA or SGEMM_PATH_TF32X3; 0 = no kernel (m or n is 0) */
    int kernel;        /* 0 FFMA GEMM kernel, 1 C = beta*C scale kernel, 2 3xTF32 tensor-core
                          GEMM (after one split launch when an operand is not read as stored) */
    int bm, bn, bk;    /* CTA tile (rows of C, columns of C, k per pipeline stage)             */
    int rm, rn;        /* per-thread register tile of C (FFMA path; 0 otherwise)               */
    int threads;       /* threads per CTA                                                      */
    int stages;        /* shared-memory pipeline depth                                         */
    int grid;          /* CTAs launched (tiles * split_k; 2 * tiles for CTA pairs)             */
    int tiles;         /* output tiles = ceil(m/bm) * ceil(n/bn)                               */
    int k_tiles;       /* pipeline stages consumed per tile = ceil(k/bk)                       */
    int smem_bytes;    /* dynamic shared memory per CTA                                        */
    int b_vec;         /* 1: B loaded 16 bytes at a time / by TMA                              */
    int c_vec;         /* 1: C read and written 16 bytes at a time                             */
    int group_m;       /* tile rows per raster group (L2 reuse)                                */
    int split_k;       /* CTAs sharing one tile along k (a thread-block cluster; 1 = no split) */
    int op_a, op_b;    /* SGEMM_OP_N / SGEMM_OP_T of the problem planned                      */
    int a_vec;         /* 1: A (stored k x m) loaded 16 bytes at a time (FFMA path)            */
    int a_in_kernel;   /* 1: the tensor-core GEMM reads A as stored (TMA) and splits it itself */
                       /*    (in four row phases when its rows are not 16 bytes apart)      */
    int trans;         /* 1: tensor-core tiles of C^T = B^T A^T (n <= 128; bm = 256, bn = 128) */
    int stream_k;      /* > 0: stream-K over this many CTAs (grid): the full waves as whole   */
                       /*      tiles, the rest shared out by k slabs (equal runs, or sk_parts  */
                       /*      parts a tile); partial tiles meet in a workspace                */
    int b_in_kernel;   /* 1: the same for B (no split pass, no scratch for that operand)       */
    int pair;          /* 1: CTA pairs (cta_group::2) compute 256 x 256 tiles, 2 CTAs per tile */
    int persistent;    /* 1: grid CTAs take whole tiles g, g + grid, ... in turn (more than a wave) */
    int sk_parts;      /* stream-K, >= 2: the tiles left after the full waves are each cut into */
                       /*      sk_parts equal k ranges (one per CTA) instead of equal runs    */
} sgemm_plan;

int sgemm_plan_for(int m, int n, int k, float alpha,
                   const float *A, int lda, const float *B, int ldb,
                   float beta, const float *C, int ldc, int path, int num_sms,
                   sgemm_plan *plan);

/*
 * Device-side status word of the tensor-core path on the current device: its
 * pipeline waits are bounded, and a wait that runs out sets a non-zero code
 * (the kernel then abandons its tile instead of hanging).  Synchronises the
 * device, copies the word to *flag and, when `clear` is non-zero, resets it.
 * The first code recorded is kept (per group of kernels the library
 * compiles together; the first group's non-zero code is returned): 0x201
 * the TMA producer waited for a free
 * ring slot, 0x202 the MMA issuer for a loaded (or split) slab, 0x203 the
 * accumulator warps for a finished chunk, 0x204 a wait while draining after
 * an earlier timeout, 0x205 the MMA issuer for a free TMEM buffer, 0x206 the
 * splitter warps for a loaded slab.  Each means the result of that call is
 * not valid.  0x207 is recorded only by sgemm_selftest_wait.  0x208 (checked
 * builds only, see sgemm_bounds_line): a kernel computed an index outside the
 * buffer it was about to access, and skipped that access.
 */
int sgemm_device_status(int *flag, int clear);

/*
 * Checked builds.  The library can be compiled with SGEMM_GB300_CHECKED
 * defined (the Python build makes it as a second library,
 * libsgemm_gb300_checked_<arch>.so): every kernel then tests each global and
 * shared-memory index it computes against the buffer it addresses (C's m x n
 * window with row pitch ldc, each operand's rows x k or k x rows window, the
 * split arrays, the stream-K workspace, each shared-memory region) before
 * the access.  A failed test skips the access -- nothing outside a buffer is
 * read or written, no kernel traps -- and records 0x208 in the device status
 * word and the source line of the test.  The checks cost time; the release
 * library has none of them.
 *
 * sgemm_bounds_line: synchronises the device and copies the source line of
 * the first failed test to *line (0: none; always 0 in a release build);
 * `clear` non-zero resets it and the status word (as sgemm_device_status's
 * `clear` resets both).  Status 1: line is NULL; 100: CUDA error.
 *
 * sgemm_selftest_bounds: checked builds run one store whose index test is
 * made to fail (the store is skipped), so 0x208 is recorded in the status
 * word (unless an earlier code is kept there) and *line receives the line of
 * the first failed test; returns 0.  A release build returns
 * SGEMM_STATUS_UNSUPPORTED and runs nothing.  Status 1: line is NULL; 100:
 * CUDA error.
 */
int sgemm_bounds_line(int *line, int clear);
int sgemm_selftest_bounds(int *line);

/*
 * Diagnostic for the failure-reporting path: runs one bounded wait on a
 * shared-memory barrier that nothing signals, through the same bounded-wait
 * routine as the GEMM's pipeline waits.  It gives up after `limit_ns`
 * nanoseconds (1 .. 10^10), records 0x207 in the device status word (unless
 * an earlier code is kept there) and returns; the context stays usable.
 * Synchronises the device; *gave_up (host pointer) = 1 when the wait ran
 * out.  Status 1: limit_ns out of range; 2: gave_up is NULL; 100: CUDA error.
 *
 * Fault injection for tests: with the environment variable
 * SGEMM_GB300_FAIL_ALLOC set, the tensor-core path's scratch allocation
 * reports cudaErrorMemoryAllocation without being attempted, so a call that
 * needs scratch returns 100 before launching anything (C is not written);
 * a call that needs none runs as usual.
 */
int sgemm_selftest_wait(unsigned long long limit_ns, int *gave_up);

/* Library version string, e.g. "sgemm_gb300 0.1 (sm_103a)"; a checked build
 * ends in ", checked)". */
const char *sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
