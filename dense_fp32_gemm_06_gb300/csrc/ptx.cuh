// Inline-PTX helpers for sm_103a: asynchronous copies, mbarriers, TMA.
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

namespace sgemm_gb300 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- cp.async

// 4-byte asynchronous copy; `src_bytes` 0 fills the destination with zero
// and reads nothing.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// 16-byte asynchronous copy bypassing L1; bytes past `src_bytes` are zero.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// One arrival on an mbarrier of another CTA of the cluster (`bar_cluster`:
// a shared::cluster address, from mapa), releasing this thread's earlier
// writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(bar_cluster) : "memory");
}

// Asynchronous bulk copy of `bytes` (a multiple of 16) from this CTA's
// shared memory to another CTA of the cluster (`dst_cluster`, a
// shared::cluster address); its completion is signalled as transaction
// bytes on the mbarrier at `bar_cluster` in the destination CTA.  The
// issuing thread does not wait for it.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                                  uint32_t bar_cluster) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                     dst_cluster),
                 "r"(src_cta), "r"(bytes), "r"(bar_cluster)
                 : "memory");
}

// try_wait with acquire at cluster scope: for barriers that other CTAs of
// the cluster arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Asks for the 128-byte line holding `p` to be brought into L2 (a hint:
// nothing waits for it).
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(reinterpret_cast<uint64_t>(p)));
}

// The same for `bytes` (a multiple of 16) from `p` (16-byte aligned), by the
// bulk-copy engine: one instruction for a whole buffer.
__device__ __forceinline__ void bulk_prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Status word written by bounded waits that gave up (0 = never).  Each
// translation unit of the library has its own (internal linkage: the units
// are compiled apart), read through unit_status below.
static __device__ int g_sgemm_status;

// ---------------------------------------------------------------- checked builds
// Compiled with SGEMM_GB300_CHECKED, the kernels test each global and
// shared-memory index they compute against its buffer before the access
// (SG_IN(condition)): a failed test skips that access, records kStatusBounds
// in the status word and the source line of the test in g_sgemm_bad_line,
// and the call's results are then not valid.  No test traps or returns
// early: barriers and waits run as usual, the context stays usable.
// Without SGEMM_GB300_CHECKED, SG_IN(c) is `true` and the tests compile away.
constexpr int kStatusBounds = 0x208;
static __device__ int g_sgemm_bad_line;

#ifdef SGEMM_GB300_CHECKED
#define SG_CHECK_FN static __device__ __noinline__   // one copy of each test per unit: short compile times
#else
#define SG_CHECK_FN static __device__ __forceinline__
#endif

SG_CHECK_FN bool bounds_ok(bool ok, int line) {
    if (!ok) {
        atomicCAS(&g_sgemm_status, 0, kStatusBounds);
        atomicCAS(&g_sgemm_bad_line, 0, line);
    }
    return ok;
}

#ifdef SGEMM_GB300_CHECKED
#define SG_IN(cond) (::sgemm_gb300::bounds_ok((cond), __LINE__))
#else
#define SG_IN(cond) (true)
#endif

// Whether `p` addresses an element (r, c) of the rows x cols matrix at
// `base` (row pitch ld) whose row holds the n elements from c on.
SG_CHECK_FN bool in_matrix(const float *p, int n, const float *base, long long ld, long long rows, long long cols) {
    const long long off = p - base;
    if (off < 0 || ld <= 0) return false;
    const long long r = off / ld, c = off - r * ld;
    return r < rows && c + n <= cols;
}

// Bounded wait for the phase of parity `parity` of `bar`: gives up after
// `limit_ns` nanoseconds, records `code` in g_sgemm_status and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int code,
                                          uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicCAS(&g_sgemm_status, 0, code);
            return false;
        }
    }
    return true;
}

// The same, acquiring at cluster scope (a barrier other CTAs arrive on).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, int code,
                                                  uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_cluster(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicCAS(&g_sgemm_status, 0, code);
            return false;
        }
    }
    return true;
}

// This translation unit's status word and failed-test line (host side;
// synchronise first): copied to *status / *line (either may be NULL), and
// reset when `clear` is set.
static inline cudaError_t unit_status(int *status, int *line, bool clear) {
    cudaError_t e = cudaSuccess;
    if (status) e = cudaMemcpyFromSymbol(status, g_sgemm_status, sizeof(int));
    if (e == cudaSuccess && line) e = cudaMemcpyFromSymbol(line, g_sgemm_bad_line, sizeof(int));
    if (e == cudaSuccess && clear) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_sgemm_status, &zero, sizeof(int));
        if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_sgemm_bad_line, &zero, sizeof(int));
    }
    return e;
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void *desc) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(desc)) : "memory");
}

// 2-D tiled TMA load of the box at (x = innermost coordinate, y) into shared
// memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *desc, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 3-D tiled TMA load of the box at (x, y, z) (x innermost).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *desc, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(desc)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Programmatic dependent launch: a kernel launched as the dependent of the
// previous kernel in its stream may start before that kernel completes;
// griddep_wait() blocks the calling thread until the previous kernel has
// completed and its memory operations are visible (a no-op for a kernel
// launched normally).  griddep_launch_dependents() lets the next kernel in
// the stream, if launched as a dependent, start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

}  // namespace sgemm_gb300
