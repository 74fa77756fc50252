// Inline-PTX wrappers for the 5th-generation tensor core (tcgen05) on
// sm_103a: tensor-memory allocation, MMA issue and commit, TMEM -> register
// loads, the tcgen05 fences, and the shared-memory matrix descriptor.
#pragma once
#include <cstdint>

namespace sgemm_gb300 {
namespace tc {

// ---------------------------------------------------------------- TMEM

// Allocates `ncols` (power of two, >= 32) tensor-memory columns for this CTA
// and writes the base address to shared memory at `dst_smem`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

// Whole warp.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

// The same for a CTA pair (cta_group::2): one warp of each of the two peer
// CTAs executes it, and the columns are allocated (freed) in both CTAs'
// tensor memory at the same address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (TMA, tensor core).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// ---------------------------------------------------------------- MMA

// D[tmem] (+)= A[smem] * B[smem]^T, kind::tf32, issued by one thread.
// `accumulate` == 0 overwrites D.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The CTA pair's MMA (cta_group::2), issued by one thread of the even CTA:
// A's rows are split between the two CTAs (M / 2 in each, same shared-memory
// offset), B's between them likewise (N / 2 in each), and each CTA's tensor
// memory receives its M / 2 rows of D, all N columns.
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One arrival on the mbarrier at shared-memory offset `bar` in every CTA of
// `cta_mask` (bit i = cluster rank i) once the pair MMAs this thread issued
// have completed.
__device__ __forceinline__ void commit_pair(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

// The mbarrier at `bar` (shared, 32-bit address) receives one arrival when
// every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}

// Instruction descriptor of kind::tf32 with FP32 accumulation.  Bit fields:
// [4,6) D format (1 = F32), [7,10) A format and [10,13) B format (2 = TF32),
// 15 / 16 A / B major (0 = K-major: rows of the operand hold consecutive k;
// 1 = MN-major: rows hold consecutive m / n), [17,23) N >> 3, [24,29) M >> 4.
template <int M, int N, bool A_MN = false, bool B_MN = false>
__host__ __device__ constexpr uint32_t idesc_tf32_f32() {
    static_assert(M == 64 || M == 128 || M == 256, "M: 64 or 128 (one CTA), 128 or 256 (a CTA pair)");
    static_assert(N % 16 == 0 && N >= 16 && N <= 256, "N");
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(A_MN) << 15) | (uint32_t(B_MN) << 16) |
           (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major operand stored as rows of
// 64 bytes (16 TF32 values) with the 64-byte swizzle: 8-row groups are
// 512 bytes apart (stride byte offset); the leading byte offset is unused
// for swizzled K-major layouts.  Bits: [0,14) start >> 4, [16,30) LBO >> 4,
// [32,46) SBO >> 4, [46,48) version 1, [61,64) layout (4 = 64B swizzle).
// The k step of 8 values inside a row is a 32-byte advance of the start.
__device__ __forceinline__ uint64_t desc_kmajor_sw64(uint32_t smem_addr) {
    uint64_t d = (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)((512u >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)4u << 61;
    return d;
}

// Descriptor of an MN-major operand (rows of the operand = consecutive m or
// n in memory) as TMA writes it with the 128-byte swizzle of 32-byte atoms
// (CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B: 32-byte chunks permuted within each
// 128-byte line), layout code 1 here.  A slab is stored as boxes of
// 32 operand rows (one 128-byte line per k) by 16 k, box j of the tile at
// j * 2048 bytes.  Fields, as measured on GB300 with identity products
// whose every output names the element it was read from: the leading byte
// offset is the distance between 32-row atoms along m / n (2048 here), the
// stride byte offset the distance between groups of 4 k lines (512); the k
// step of 8 values is a 1024-byte advance of the start.  (With the 16-byte
// 128-byte swizzle, layout code 2, an MN-major TF32 operand multiplied as
// zeros, whatever the offsets.)
__device__ __forceinline__ uint64_t desc_mnmajor_sw128_32b(uint32_t smem_addr) {
    uint64_t d = (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((2048u >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((512u >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)1u << 61;
    return d;
}

// ---------------------------------------------------------------- TMEM -> registers

// 32 consecutive 32-bit columns of this thread's TMEM lane (lanes of warp w
// are 32*(w%4) .. 32*(w%4)+31).  Whole warp; follow with wait_ld().
__device__ __forceinline__ void ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.  Whole warp.
__device__ __forceinline__ void ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

// ---------------------------------------------------------------- thread-block clusters

// Rank of this CTA in its cluster and the cluster's size (0 and 1 when the
// kernel is launched without clusters).
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; orders shared-memory writes
// before the barrier with reads after it, across the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n"
        "barrier.cluster.wait.acquire.aligned;\n" ::
            : "memory");
}

// The two halves of a cluster barrier: an arrival that orders nothing (for
// a thread whose earlier accesses to other CTAs' shared memory are loads
// whose values it has already used), and the wait for every thread of the
// cluster to have arrived.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory"); }

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// ---------------------------------------------------------------- TF32 rounding

// Rounds an FP32 value to TF32 (10 explicit mantissa bits), to nearest with
// ties away from zero; the result is an FP32 bit pattern whose low 13 bits
// are zero.
__device__ __forceinline__ float round_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

}  // namespace tc
}  // namespace sgemm_gb300
