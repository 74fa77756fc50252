// CUDA-core FFMA SGEMM for sm_103a: C = alpha*A*B + beta*C, row-major FP32.
//
// Design (the two-level blocking of hatrix.site "GEMM优化原理", sections
// 基于 shared memory 计算 and 基于 register 计算, re-sized for GB300):
//
//  * one CTA owns a BM x BN tile of C; tiles are visited in groups of
//    `group_m` tile rows so that CTAs resident at the same time share A and
//    B panels in L2 (the grouped block order of blog.lightlisten.com
//    "gemm优化", section "Swizzle 增强L2缓存命中");
//  * K is consumed in BK-deep slabs through a STAGES-deep ring of shared
//    memory filled by cp.async (the multi-buffer pipeline of aerisun.top
//    "GPU 访存与计算优化", section 数据搬运与计算流水线): a slab is waited for
//    before use, and a buffer is refilled only after the barrier that proves
//    every warp has finished reading it;
//  * A is scattered into shared memory transposed, as [BK][BM+4], by 4-byte
//    copies: each warp copies a 4-row x 8-column patch (four full 32-byte
//    sectors of global memory) and, because the row pitch BM+4 is 4 banks
//    past a multiple of 32, its 32 stores land in 32 different banks.  The
//    same 4-byte copies serve any lda and any alignment and zero-fill the m
//    and k tails (out-of-range inputs are zero and every thread reaches every
//    barrier: aerisun.top, section "Shared Tiling 与 block 内复用");
//  * B is copied row by row as [BK][BN], 16 bytes per copy when its rows
//    are 16-byte aligned, else 4 bytes; partial 16-byte copies zero-fill the
//    n tail;
//  * each thread accumulates a TM x TN register tile made of 4 x 4 blocks:
//    rows a_off + 32g + {0..3}, columns b_off + 16h + {0..3}.  Every fragment
//    read is one 16-byte shared load (LDS.128), and a warp (8 x 4 lanes) reads
//    8 contiguous 16-byte words of one A row and 4 of one B row: a single
//    wavefront each, no bank conflict.  Per k a thread issues
//    (TM + TN) / 4 LDS.128 for TM*TN FFMA (bk small iterations of rm*rn FFMA
//    each, hatrix.site section 基于 register 计算); fragments for k+1 are
//    loaded while k is multiplied (ping-pong registers);
//  * the epilogue forms alpha*acc + beta*C (C not read when beta == 0) and
//    stores 16 bytes at a time where C rows are 16-byte aligned, predicated
//    element by element at the m and n edges.
#pragma once
#include <cstdint>

#include "ptx.cuh"
#include "raster.cuh"

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

template <int BM_, int BN_, int BK_, int STAGES_, int TM_, int TN_, int MIN_BLOCKS_>
struct Config {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, STAGES = STAGES_, TM = TM_, TN = TN_;
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_;
    static constexpr int WARP_M = 8 * TM;            // rows of C per warp (8 lanes x TM)
    static constexpr int WARP_N = 4 * TN;            // columns of C per warp (4 lanes x TN)
    static constexpr int WARPS_M = BM / WARP_M;
    static constexpr int WARPS_N = BN / WARP_N;
    static constexpr int WARPS = WARPS_M * WARPS_N;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int A_LD = BM + 4;              // floats per k-row of the transposed A slab
    static constexpr int A_STAGE = BK * A_LD;        // floats
    static constexpr int B_STAGE = BK * BN;          // floats
    static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
    static constexpr int A_CHUNKS = (BM / 4) * (BK / 8);   // 32-element patches per slab
    static constexpr int A_PER_WARP = A_CHUNKS / WARPS;
    static constexpr int B_VEC_PER_THREAD = BK * BN / 4 / THREADS;
    static constexpr int B_SCALAR_PER_THREAD = BK * BN / THREADS;

    static_assert(TM % 4 == 0 && TN % 4 == 0, "register tile is made of 4 x 4 blocks");
    static_assert(BM % WARP_M == 0 && BN % WARP_N == 0, "warps tile the CTA tile");
    static_assert(BK % 8 == 0 && BM % 4 == 0, "A patches are 4 rows x 8 columns");
    static_assert(A_CHUNKS % WARPS == 0, "A patches split evenly over warps");
    static_assert((BK * BN / 4) % THREADS == 0, "B float4s split evenly over threads");
    static_assert((A_LD % 32) == 4, "A pitch must sit 4 banks past a multiple of 32");
    static_assert((A_LD * 4) % 16 == 0, "A rows must keep 16-byte fragment alignment");
    static_assert(STAGES >= 2, "at least double buffering");
};

// Per-thread state of the slab loader.  Every address a thread copies from
// is fixed up to the slab offset k0, so it is computed once: the A rows of a
// thread are A_ROW_STEP apart, its B rows B_ROW_STEP apart.  Interior slabs
// (the whole BM x BK / BK x BN box inside the matrices) take copies with no
// predicate; edge slabs test every element and zero-fill.
template <class Cfg, bool B_VEC>
struct SlabLoader {
    static constexpr int A_ROW_STEP = (Cfg::WARPS / (Cfg::BK / 8)) * 4;
    static constexpr int B_ROWS_PER_PASS = B_VEC ? Cfg::THREADS / (Cfg::BN / 4) : Cfg::THREADS / Cfg::BN;
    static_assert(Cfg::WARPS % (Cfg::BK / 8) == 0, "A patches of one thread share a column");

    const float *a_src;      // A + (m0 + row0) * lda + kc   (row clamped into the matrix)
    const float *b_src;      // B + brow0 * ldb + n0 + bcol  (clamped)
    uint32_t a_dst, b_dst;   // shared byte offsets inside a stage
    int a_row0, a_kc, b_row0, b_col;
    long long a_step, b_step;   // A_ROW_STEP * lda, B_ROWS_PER_PASS * ldb (elements)
    bool interior_mn;

    __device__ __forceinline__ SlabLoader(const GemmArgs &p, int m0, int n0, int tid) {
        const int warp = tid >> 5, lane = tid & 31;
        a_row0 = (warp / (Cfg::BK / 8)) * 4 + (lane >> 3);
        a_kc = (warp % (Cfg::BK / 8)) * 8 + (lane & 7);
        const int ar = min(m0 + a_row0, p.m - 1);
        a_src = p.A + (long long)ar * p.lda + a_kc;
        a_step = (long long)A_ROW_STEP * p.lda;
        a_dst = (uint32_t)(a_kc * Cfg::A_LD + a_row0) * 4u;
        if constexpr (B_VEC) {
            b_row0 = tid / (Cfg::BN / 4);
            b_col = (tid % (Cfg::BN / 4)) * 4;
        } else {
            b_row0 = tid / Cfg::BN;
            b_col = tid % Cfg::BN;
        }
        b_src = p.B + (long long)b_row0 * p.ldb + min(n0 + b_col, p.n - 1);
        b_step = (long long)B_ROWS_PER_PASS * p.ldb;
        b_dst = (uint32_t)(b_row0 * Cfg::BN + b_col) * 4u;
        interior_mn = m0 + Cfg::BM <= p.m && n0 + Cfg::BN <= p.n;
    }

    __device__ __forceinline__ void load(const GemmArgs &p, uint32_t As, uint32_t Bs, int m0, int n0, int k0) const {
        if (interior_mn && k0 + Cfg::BK <= p.k) {
            const float *a = a_src + k0;
#pragma unroll
            for (int j = 0; j < Cfg::A_PER_WARP; ++j, a += a_step)
                cp_async_4(As + a_dst + j * A_ROW_STEP * 4, a, 4u);
            const float *b = b_src + (long long)k0 * p.ldb;
            if constexpr (B_VEC) {
#pragma unroll
                for (int j = 0; j < Cfg::B_VEC_PER_THREAD; ++j, b += b_step)
                    cp_async_16(Bs + b_dst + j * B_ROWS_PER_PASS * Cfg::BN * 4, b, 16u);
            } else {
#pragma unroll
                for (int j = 0; j < Cfg::B_SCALAR_PER_THREAD; ++j, b += b_step)
                    cp_async_4(Bs + b_dst + j * B_ROWS_PER_PASS * Cfg::BN * 4, b, 4u);
            }
            return;
        }
        // edge slab: predicate every copy, zero-fill what lies outside
        {
            const bool k_ok = k0 + a_kc < p.k;
            const float *a = a_src + (k_ok ? k0 : 0);
#pragma unroll
            for (int j = 0; j < Cfg::A_PER_WARP; ++j) {
                const bool ok = k_ok && m0 + a_row0 + j * A_ROW_STEP < p.m;
                cp_async_4(As + a_dst + j * A_ROW_STEP * 4, ok ? a + j * a_step : p.A, ok ? 4u : 0u);
            }
        }
        if constexpr (B_VEC) {
            const int left = p.n - (n0 + b_col);
            const uint32_t bytes = left >= 4 ? 16u : (left > 0 ? 4u * left : 0u);
#pragma unroll
            for (int j = 0; j < Cfg::B_VEC_PER_THREAD; ++j) {
                const int kr = k0 + b_row0 + j * B_ROWS_PER_PASS;
                const uint32_t nb = kr < p.k ? bytes : 0u;
                cp_async_16(Bs + b_dst + j * B_ROWS_PER_PASS * Cfg::BN * 4,
                            nb ? b_src + (long long)(k0 + j * B_ROWS_PER_PASS) * p.ldb : p.B, nb);
            }
        } else {
            const bool n_ok = n0 + b_col < p.n;
#pragma unroll
            for (int j = 0; j < Cfg::B_SCALAR_PER_THREAD; ++j) {
                const int kr = k0 + b_row0 + j * B_ROWS_PER_PASS;
                const bool ok = n_ok && kr < p.k;
                cp_async_4(Bs + b_dst + j * B_ROWS_PER_PASS * Cfg::BN * 4,
                           ok ? b_src + (long long)(k0 + j * B_ROWS_PER_PASS) * p.ldb : p.B, ok ? 4u : 0u);
            }
        }
    }
};

template <class Cfg, bool B_VEC, bool C_VEC>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_BLOCKS) ffma_sgemm_kernel(const GemmArgs p) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int TM = Cfg::TM, TN = Cfg::TN, A_LD = Cfg::A_LD;
    constexpr int GM = TM / 4, GN = TN / 4;   // 4 x 4 blocks per thread

    extern __shared__ __align__(16) float smem[];
    float *const As = smem;                            // [STAGES][BK][A_LD]
    float *const Bs = smem + STAGES * Cfg::A_STAGE;    // [STAGES][BK][BN]

    const int tid = threadIdx.x;
    int tm, tn;
    raster_tile(blockIdx.x, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * BM, n0 = tn * BN;
    const int KT = (p.k + BK - 1) / BK;

    const int warp = tid >> 5, lane = tid & 31;
    const int a_off = (warp / Cfg::WARPS_N) * Cfg::WARP_M + (lane >> 2) * 4;
    const int b_off = (warp % Cfg::WARPS_N) * Cfg::WARP_N + (lane & 3) * 4;

    const SlabLoader<Cfg, B_VEC> loader(p, m0, n0, tid);
    const uint32_t As_u32 = smem_u32(As), Bs_u32 = smem_u32(Bs);

    // prologue: slabs 0 .. STAGES-2 in flight
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < KT) loader.load(p, As_u32 + s * Cfg::A_STAGE * 4, Bs_u32 + s * Cfg::B_STAGE * 4, m0, n0, s * BK);
        cp_async_commit();
    }

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    for (int kt = 0; kt < KT; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();   // slab kt visible to all; slab kt-1 fully consumed
        {
            const int nk = kt + STAGES - 1;
            if (nk < KT) {
                const int s = nk % STAGES;
                loader.load(p, As_u32 + s * Cfg::A_STAGE * 4, Bs_u32 + s * Cfg::B_STAGE * 4, m0, n0, nk * BK);
            }
            cp_async_commit();
        }
        const int s = kt % STAGES;
        const float *as = As + s * Cfg::A_STAGE + a_off;
        const float *bs = Bs + s * Cfg::B_STAGE + b_off;

        float4 fa[2][GM], fb[2][GN];
#pragma unroll
        for (int g = 0; g < GM; ++g) fa[0][g] = *reinterpret_cast<const float4 *>(as + 32 * g);
#pragma unroll
        for (int h = 0; h < GN; ++h) fb[0][h] = *reinterpret_cast<const float4 *>(bs + 16 * h);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const int cur = kk & 1;
            if (kk + 1 < BK) {
                const int nxt = cur ^ 1;
#pragma unroll
                for (int g = 0; g < GM; ++g)
                    fa[nxt][g] = *reinterpret_cast<const float4 *>(as + (kk + 1) * A_LD + 32 * g);
#pragma unroll
                for (int h = 0; h < GN; ++h)
                    fb[nxt][h] = *reinterpret_cast<const float4 *>(bs + (kk + 1) * BN + 16 * h);
            }
            float a[TM], b[TN];
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                a[4 * g + 0] = fa[cur][g].x;
                a[4 * g + 1] = fa[cur][g].y;
                a[4 * g + 2] = fa[cur][g].z;
                a[4 * g + 3] = fa[cur][g].w;
            }
#pragma unroll
            for (int h = 0; h < GN; ++h) {
                b[4 * h + 0] = fb[cur][h].x;
                b[4 * h + 1] = fb[cur][h].y;
                b[4 * h + 2] = fb[cur][h].z;
                b[4 * h + 3] = fb[cur][h].w;
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    cp_async_wait<0>();

    // ---- epilogue
    const float alpha = p.alpha, beta = p.beta;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + a_off + 32 * (i / 4) + (i % 4);
        if (row >= p.m) continue;
        float *crow = p.C + (long long)row * p.ldc;
#pragma unroll
        for (int h = 0; h < GN; ++h) {
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

// The configuration the library launches.
using Default = Config<128, 128, 32, 3, 8, 8, 2>;

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
