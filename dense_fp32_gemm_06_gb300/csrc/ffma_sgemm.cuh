// CUDA-core FFMA SGEMM for sm_103a: C = alpha*A*B + beta*C, row-major FP32.
//
// Design (the two-level blocking of hatrix.site "GEMM优化原理", sections
// 基于 shared memory 计算 and 基于 register 计算, re-sized for GB300):
//
//  * one CTA of 256 threads owns a BM x BN = 128 x 128 tile of C; tiles are
//    visited in groups of `group_m` tile rows so that CTAs resident at the
//    same time share A and B panels in L2 (the grouped block order of
//    blog.lightlisten.com "gemm优化", section "Swizzle 增强L2缓存命中");
//  * K is consumed in BK = 16 slabs through a STAGES-deep ring of shared
//    memory filled by cp.async (the multi-buffer pipeline of aerisun.top
//    "GPU 访存与计算优化", section 数据搬运与计算流水线): a slab is waited for
//    before use, and a buffer is refilled only after the barrier that proves
//    every warp has finished reading it;
//  * A is scattered into shared memory transposed, as [BK][BM+4], by 4-byte
//    copies: each warp copies a 4-row x 8-column patch (four full 32-byte
//    sectors of global memory) and, because the row pitch BM+4 is 4 banks
//    past a multiple of 32, its 32 stores land in 32 different banks.  The
//    same 4-byte copies serve any lda and any alignment and zero-fill the m
//    and k tails (out-of-range inputs are zero, every thread reaches every
//    barrier: aerisun.top, section "Shared Tiling 与 block 内复用");
//  * B is copied row by row as [BK][BN], 16 bytes per copy when its rows
//    are 16-byte aligned, else 4 bytes; partial 16-byte copies zero-fill the
//    n tail;
//  * each thread accumulates an 8 x 8 register tile, split as 2 x 2 blocks
//    of 4 x 4 so that every fragment read is one 16-byte shared load (LDS.128)
//    and a warp's A (resp. B) fragment read touches 8 (resp. 4) contiguous
//    16-byte words of one shared row: one wavefront, no bank conflict.  Per k
//    a thread issues 4 LDS.128 for 64 FFMA (bk small iterations of rm*rn
//    FFMA each, hatrix.site section 基于 register 计算).  Fragments for k+1
//    are loaded while k is multiplied (ping-pong registers);
//  * the epilogue forms alpha*acc + beta*C (C not read when beta == 0) and
//    stores 16 bytes at a time where C rows are 16-byte aligned, predicated
//    element by element at the m and n edges.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace sgemm_gb300 {

struct GemmArgs {
    int m, n, k;
    float alpha, beta;
    const float *A;
    long long lda;
    const float *B;
    long long ldb;
    float *C;
    long long ldc;
    int tiles_m, tiles_n;
    int group_m;
};

namespace ffma {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 16;
constexpr int STAGES = 4;
constexpr int THREADS = 256;
constexpr int RM = 8;
constexpr int RN = 8;
constexpr int A_LD = BM + 4;           // floats per k-row of the transposed A slab
constexpr int A_STAGE = BK * A_LD;     // floats
constexpr int B_STAGE = BK * BN;       // floats
constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;

static_assert(BM * BK == 8 * THREADS, "A loader: 8 four-byte copies per thread per slab");
static_assert(BK * BN == 8 * THREADS, "B loader: 8 floats per thread per slab");
static_assert((A_LD % 32) == 4, "A pitch must sit 4 banks past a multiple of 32");
static_assert((A_LD * 4) % 16 == 0, "A rows must keep 16-byte fragment alignment");

// Maps a linear CTA index onto (tile row, tile column): tiles are taken
// column by column inside groups of `group_m` tile rows.
__device__ __forceinline__ void raster_tile(int tile, int tiles_m, int tiles_n, int group_m,
                                            int &tm, int &tn) {
    const int per_group = group_m * tiles_n;
    const int group = tile / per_group;
    const int first_m = group * group_m;
    const int rows = min(tiles_m - first_m, group_m);
    const int in_group = tile - group * per_group;
    tm = first_m + in_group % rows;
    tn = in_group / rows;
}

template <bool B_VEC>
__device__ __forceinline__ void load_slab(const GemmArgs &p, float *As, float *Bs, int m0, int n0,
                                          int k0, int tid) {
    const int warp = tid >> 5, lane = tid & 31;
    // ---- A: 8 rows (16 apart) x one column per thread, stored transposed.
    {
        const int r0 = (warp >> 1) * 4 + (lane >> 3);   // 0..15
        const int kc = (warp & 1) * 8 + (lane & 7);     // 0..15
        const int kk = k0 + kc;
        const bool k_ok = kk < p.k;
        const uint32_t dst0 = smem_u32(As + kc * A_LD + r0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int row = m0 + 16 * j + r0;
            const bool ok = k_ok && row < p.m;
            const float *src = ok ? p.A + (long long)row * p.lda + kk : p.A;
            cp_async_4(dst0 + 16 * j * 4, src, ok ? 4u : 0u);
        }
    }
    // ---- B: [BK][BN], row-major like global memory.
    if constexpr (B_VEC) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int row = j * 8 + warp;   // 0..15
            const int col = n0 + lane * 4;
            const int kr = k0 + row;
            int bytes = 0;
            if (kr < p.k) {
                const int left = p.n - col;
                bytes = left >= 4 ? 16 : (left > 0 ? left * 4 : 0);
            }
            const float *src = bytes ? p.B + (long long)kr * p.ldb + col : p.B;
            cp_async_16(smem_u32(Bs + row * BN + lane * 4), src, (uint32_t)bytes);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int row = 2 * j + (tid >> 7);   // 0..15
            const int c = tid & 127;
            const int kr = k0 + row, col = n0 + c;
            const bool ok = kr < p.k && col < p.n;
            const float *src = ok ? p.B + (long long)kr * p.ldb + col : p.B;
            cp_async_4(smem_u32(Bs + row * BN + c), src, ok ? 4u : 0u);
        }
    }
}

template <bool B_VEC, bool C_VEC>
__global__ void __launch_bounds__(THREADS, 2) ffma_sgemm_kernel(const GemmArgs p) {
    extern __shared__ __align__(16) float smem[];
    float *const As = smem;                     // [STAGES][BK][A_LD]
    float *const Bs = smem + STAGES * A_STAGE;  // [STAGES][BK][BN]

    const int tid = threadIdx.x;
    int tm, tn;
    raster_tile(blockIdx.x, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * BM, n0 = tn * BN;
    const int KT = (p.k + BK - 1) / BK;

    const int warp = tid >> 5, lane = tid & 31;
    const int a_off = (warp >> 2) * 64 + (lane >> 2) * 4;   // thread rows: a_off+{0..3}, a_off+32+{0..3}
    const int b_off = (warp & 3) * 32 + (lane & 3) * 4;     // thread cols: b_off+{0..3}, b_off+16+{0..3}

    // prologue: slabs 0 .. STAGES-2 in flight
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < KT) load_slab<B_VEC>(p, As + s * A_STAGE, Bs + s * B_STAGE, m0, n0, s * BK, tid);
        cp_async_commit();
    }

    float acc[RM][RN];
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int j = 0; j < RN; ++j) acc[i][j] = 0.f;

    for (int kt = 0; kt < KT; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();   // slab kt visible to all; slab kt-1 fully consumed
        {
            const int nk = kt + STAGES - 1;
            if (nk < KT) {
                const int s = nk % STAGES;
                load_slab<B_VEC>(p, As + s * A_STAGE, Bs + s * B_STAGE, m0, n0, nk * BK, tid);
            }
            cp_async_commit();
        }
        const int s = kt % STAGES;
        const float *as = As + s * A_STAGE + a_off;
        const float *bs = Bs + s * B_STAGE + b_off;

        float4 fa[2][2], fb[2][2];
        fa[0][0] = *reinterpret_cast<const float4 *>(as);
        fa[0][1] = *reinterpret_cast<const float4 *>(as + 32);
        fb[0][0] = *reinterpret_cast<const float4 *>(bs);
        fb[0][1] = *reinterpret_cast<const float4 *>(bs + 16);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const int cur = kk & 1;
            if (kk + 1 < BK) {
                const int nxt = cur ^ 1;
                fa[nxt][0] = *reinterpret_cast<const float4 *>(as + (kk + 1) * A_LD);
                fa[nxt][1] = *reinterpret_cast<const float4 *>(as + (kk + 1) * A_LD + 32);
                fb[nxt][0] = *reinterpret_cast<const float4 *>(bs + (kk + 1) * BN);
                fb[nxt][1] = *reinterpret_cast<const float4 *>(bs + (kk + 1) * BN + 16);
            }
            const float a[RM] = {fa[cur][0].x, fa[cur][0].y, fa[cur][0].z, fa[cur][0].w,
                                 fa[cur][1].x, fa[cur][1].y, fa[cur][1].z, fa[cur][1].w};
            const float b[RN] = {fb[cur][0].x, fb[cur][0].y, fb[cur][0].z, fb[cur][0].w,
                                 fb[cur][1].x, fb[cur][1].y, fb[cur][1].z, fb[cur][1].w};
#pragma unroll
            for (int i = 0; i < RM; ++i)
#pragma unroll
                for (int j = 0; j < RN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    cp_async_wait<0>();

    // ---- epilogue
    const float alpha = p.alpha, beta = p.beta;
#pragma unroll
    for (int i = 0; i < RM; ++i) {
        const int row = m0 + a_off + (i < 4 ? i : 28 + i);
        if (row >= p.m) continue;
        float *crow = p.C + (long long)row * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = n0 + b_off + 16 * h;
            const float *v = &acc[i][4 * h];
            if (C_VEC && col + 3 < p.n) {
                float4 o;
                if (beta != 0.f) {
                    const float4 c = *reinterpret_cast<const float4 *>(crow + col);
                    o = make_float4(fmaf(alpha, v[0], beta * c.x), fmaf(alpha, v[1], beta * c.y),
                                    fmaf(alpha, v[2], beta * c.z), fmaf(alpha, v[3], beta * c.w));
                } else {
                    o = make_float4(alpha * v[0], alpha * v[1], alpha * v[2], alpha * v[3]);
                }
                *reinterpret_cast<float4 *>(crow + col) = o;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (col + q < p.n) {
                        crow[col + q] = beta != 0.f ? fmaf(alpha, v[q], beta * crow[col + q]) : alpha * v[q];
                    }
                }
            }
        }
    }
}

}  // namespace ffma

// C = beta * C over an m x n window (beta == 0 writes zeros without reading).
__global__ void scale_c_kernel(float *C, long long ldc, int m, int n, float beta) {
    const long long total = (long long)m * n;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long i = idx / n, j = idx - i * n;
        float *c = C + i * ldc + j;
        *c = beta != 0.f ? beta * *c : 0.f;
    }
}

}  // namespace sgemm_gb300
