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
//  * both operands land in shared memory k-major, as [BK][rows]: the rows
//    of C for A, the columns of C for B.  An operand stored with k
//    contiguous (A untransposed, B transposed) is scattered there by 4-byte
//    copies (ScatterLoader): each warp copies a 4-row x 8-column patch (four
//    full 32-byte sectors of global memory) and, because the row pitch is 4
//    banks past a multiple of 32, its 32 stores land in 32 different banks.
//    An operand stored with its rows contiguous (A transposed, B
//    untransposed) is copied row by row (DirectLoader), 16 bytes per copy
//    when its rows are 16-byte aligned, else 4 bytes.  Both serve any leading
//    dimension and alignment and zero-fill the tails (out-of-range inputs
//    are zero and every thread reaches every barrier: aerisun.top, section
//    "Shared Tiling 与 block 内复用");
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
    int c_vec;   // C rows 16-byte aligned: float4 epilogue
    // strided batch: problem blockIdx.y uses A + y*stride_a, B + y*stride_b, C + y*stride_c
    long long stride_a, stride_b, stride_c;
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

    static_assert(TM % 4 == 0 && TN % 4 == 0, "register tile is made of 4 x 4 blocks");
    static_assert(BM % WARP_M == 0 && BN % WARP_N == 0, "warps tile the CTA tile");
    static_assert(STAGES >= 2, "at least double buffering");
};

// An operand seen as a `rows` x k matrix (rows of C for A, columns of C for B).
struct Operand {
    const float *ptr;
    long long ld;
    int rows, k;
};

// Operand stored with k contiguous -- element (r, t) at ptr[r*ld + t] --
// scattered into the k-major slab [BK][R+4] by 4-byte copies: warp w copies
// 4-row x 8-column patches, one element per lane, so that global reads are
// four full 32-byte sectors and the 32 shared stores hit 32 banks (the pitch
// R+4 is 4 banks past a multiple of 32).  A thread's copies share one column
// and step ROW_STEP rows.  Interior slabs (R x BK box inside the operand)
// copy without predicates; edge slabs test each element and zero-fill.
template <int R, int BK, int THREADS>
struct ScatterLoader {
    static constexpr int WARPS = THREADS / 32;
    static constexpr int LD = R + 4;
    static constexpr int CHUNKS = (R / 4) * (BK / 8);       // 32-element patches per slab
    static constexpr int PER_THREAD = CHUNKS / WARPS;
    static constexpr int ROW_STEP = (WARPS / (BK / 8)) * 4;
    static_assert(BK % 8 == 0 && R % 4 == 0, "patches are 4 rows x 8 columns");
    static_assert(CHUNKS % WARPS == 0 && WARPS % (BK / 8) == 0, "patches split evenly, one column per thread");
    static_assert((LD % 32) == 4 && (LD * 4) % 16 == 0, "conflict-free scatter, 16-byte fragment rows");

    const float *src;   // element (r_base + row0, kc), row clamped into the operand
    long long step;     // ROW_STEP rows
    uint32_t dst;       // byte offset in the slab
    int row0, kc;
    bool interior_r;

    __device__ __forceinline__ ScatterLoader(const Operand &o, int r_base, int tid) {
        const int warp = tid >> 5, lane = tid & 31;
        row0 = (warp / (BK / 8)) * 4 + (lane >> 3);
        kc = (warp % (BK / 8)) * 8 + (lane & 7);
        src = o.ptr + (long long)min(r_base + row0, o.rows - 1) * o.ld + kc;
        step = (long long)ROW_STEP * o.ld;
        dst = (uint32_t)(kc * LD + row0) * 4u;
        interior_r = r_base + R <= o.rows;
    }

    __device__ __forceinline__ void load(const Operand &o, uint32_t slab, int r_base, int k0) const {
        if (interior_r && k0 + BK <= o.k) {
            const float *a = src + k0;
#pragma unroll
            for (int j = 0; j < PER_THREAD; ++j, a += step)
                if (SG_IN(in_matrix(a, 1, o.ptr, o.ld, o.rows, o.k) && dst + j * ROW_STEP * 4 + 4 <= BK * LD * 4))
                    cp_async_4(slab + dst + j * ROW_STEP * 4, a, 4u);
            return;
        }
        const bool k_ok = k0 + kc < o.k;
        const float *a = src + (k_ok ? k0 : 0);
#pragma unroll
        for (int j = 0; j < PER_THREAD; ++j) {
            const bool ok = k_ok && r_base + row0 + j * ROW_STEP < o.rows;
            if (SG_IN((!ok || in_matrix(a + j * step, 1, o.ptr, o.ld, o.rows, o.k)) &&
                      dst + j * ROW_STEP * 4 + 4 <= BK * LD * 4))
                cp_async_4(slab + dst + j * ROW_STEP * 4, ok ? a + j * step : o.ptr, ok ? 4u : 0u);
        }
    }
};

// Operand stored with its rows contiguous -- element (r, t) at
// ptr[t*ld + r] -- copied row by row into the slab [BK][R], 16 bytes per
// copy when VEC (base and ld 16-byte aligned), else 4 bytes; a partial
// 16-byte copy zero-fills the row tail.
template <int R, int BK, int THREADS, bool VEC>
struct DirectLoader {
    static constexpr int LD = R;
    static constexpr int W = VEC ? 4 : 1;                    // floats per copy
    static constexpr int PER_ROW = R / W;
    static constexpr int PER_THREAD = BK * PER_ROW / THREADS;
    static constexpr int ROWS_PER_PASS = THREADS / PER_ROW;
    static_assert(THREADS % PER_ROW == 0 && (BK * PER_ROW) % THREADS == 0, "copies split evenly");
    static_assert((LD * 4) % 16 == 0, "16-byte fragment rows");

    const float *src;   // element (r_base + c, kk0), column clamped into the operand
    long long step;     // ROWS_PER_PASS k-rows
    uint32_t dst;
    int kk0, c;
    bool interior_r;

    __device__ __forceinline__ DirectLoader(const Operand &o, int r_base, int tid) {
        kk0 = tid / PER_ROW;
        c = (tid % PER_ROW) * W;
        src = o.ptr + (long long)kk0 * o.ld + min(r_base + c, o.rows - 1);
        step = (long long)ROWS_PER_PASS * o.ld;
        dst = (uint32_t)(kk0 * LD + c) * 4u;
        interior_r = r_base + R <= o.rows;
    }

    __device__ __forceinline__ void load(const Operand &o, uint32_t slab, int r_base, int k0) const {
        if (interior_r && k0 + BK <= o.k) {
            const float *b = src + (long long)k0 * o.ld;
#pragma unroll
            for (int j = 0; j < PER_THREAD; ++j, b += step) {
                if (!SG_IN(in_matrix(b, W, o.ptr, o.ld, o.k, o.rows) &&
                           dst + j * ROWS_PER_PASS * LD * 4 + W * 4 <= BK * LD * 4))
                    continue;
                if constexpr (VEC)
                    cp_async_16(slab + dst + j * ROWS_PER_PASS * LD * 4, b, 16u);
                else
                    cp_async_4(slab + dst + j * ROWS_PER_PASS * LD * 4, b, 4u);
            }
            return;
        }
        uint32_t bytes;
        if constexpr (VEC) {
            const int left = o.rows - (r_base + c);
            bytes = left >= 4 ? 16u : (left > 0 ? 4u * left : 0u);
        } else {
            bytes = r_base + c < o.rows ? 4u : 0u;
        }
#pragma unroll
        for (int j = 0; j < PER_THREAD; ++j) {
            const int kr = k0 + kk0 + j * ROWS_PER_PASS;
            const uint32_t nb = kr < o.k ? bytes : 0u;
            const float *b = nb ? src + (long long)(k0 + j * ROWS_PER_PASS) * o.ld : o.ptr;
            if (!SG_IN((nb == 0 || in_matrix(b, (int)nb / 4, o.ptr, o.ld, o.k, o.rows)) &&
                       dst + j * ROWS_PER_PASS * LD * 4 + W * 4 <= BK * LD * 4))
                continue;
            if constexpr (VEC)
                cp_async_16(slab + dst + j * ROWS_PER_PASS * LD * 4, b, nb);
            else
                cp_async_4(slab + dst + j * ROWS_PER_PASS * LD * 4, b, nb);
        }
    }
};

// Shared-memory sizes of a kernel instance.
template <class Cfg, class AL, class BL>
struct Layout {
    static constexpr int A_STAGE = Cfg::BK * AL::LD;   // floats
    static constexpr int B_STAGE = Cfg::BK * BL::LD;
    static constexpr int SMEM_BYTES = Cfg::STAGES * (A_STAGE + B_STAGE) * 4;
};

// d0 += a0 * b0, d1 += a1 * b1 as one packed instruction (fma.rn.f32x2 of
// sm_100-class GPUs): each half is an IEEE round-to-nearest fused
// multiply-add, the same result as fmaf, but one issue slot does two of them.
__device__ __forceinline__ void fma2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n"
        ".reg .b64 ra, rb, rd;\n"
        "mov.b64 ra, {%2, %3};\n"
        "mov.b64 rb, {%4, %5};\n"
        "mov.b64 rd, {%0, %1};\n"
        "fma.rn.f32x2 rd, ra, rb, rd;\n"
        "mov.b64 {%0, %1}, rd;\n"
        "}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

template <class Cfg, class AL, class BL>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_BLOCKS) ffma_sgemm_kernel(const GemmArgs p) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    constexpr int TM = Cfg::TM, TN = Cfg::TN, A_LD = AL::LD, B_LD = BL::LD;
    constexpr int A_STAGE = Layout<Cfg, AL, BL>::A_STAGE, B_STAGE = Layout<Cfg, AL, BL>::B_STAGE;
    constexpr int GM = TM / 4, GN = TN / 4;   // 4 x 4 blocks per thread

    extern __shared__ __align__(16) float smem[];
    float *const As = smem;                      // [STAGES][BK][A_LD]
    float *const Bs = smem + STAGES * A_STAGE;   // [STAGES][BK][B_LD]

    const int tid = threadIdx.x;
    int tm, tn;
    raster_tile(blockIdx.x, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    const int m0 = tm * BM, n0 = tn * BN;
    const int KT = (p.k + BK - 1) / BK;

    const int warp = tid >> 5, lane = tid & 31;
    const int a_off = (warp / Cfg::WARPS_N) * Cfg::WARP_M + (lane >> 2) * 4;
    const int b_off = (warp % Cfg::WARPS_N) * Cfg::WARP_N + (lane & 3) * 4;

    const long long bz = blockIdx.y;   // problem of a strided batch
    const Operand oa{p.A + bz * p.stride_a, p.lda, p.m, p.k}, ob{p.B + bz * p.stride_b, p.ldb, p.n, p.k};
    float *const Cb = p.C + bz * p.stride_c;
    const AL la(oa, m0, tid);
    const BL lb(ob, n0, tid);
    // every fragment read below lies in its stage (the largest offsets of A's
    // and B's reads; checked builds only)
    const bool frag_ok = SG_IN(a_off + (BK - 1) * A_LD + 32 * (GM - 1) + 4 <= A_STAGE &&
                               b_off + (BK - 1) * B_LD + 16 * (GN - 1) + 4 <= B_STAGE);
    const uint32_t As_u32 = smem_u32(As), Bs_u32 = smem_u32(Bs);

    // prologue: slabs 0 .. STAGES-2 in flight
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < KT) {
            la.load(oa, As_u32 + s * A_STAGE * 4, m0, s * BK);
            lb.load(ob, Bs_u32 + s * B_STAGE * 4, n0, s * BK);
        }
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
                la.load(oa, As_u32 + s * A_STAGE * 4, m0, nk * BK);
                lb.load(ob, Bs_u32 + s * B_STAGE * 4, n0, nk * BK);
            }
            cp_async_commit();
        }
        const int s = kt % STAGES;
        const float *as = As + s * A_STAGE + a_off;
        const float *bs = Bs + s * B_STAGE + b_off;

        float4 fa[2][GM], fb[2][GN];
#pragma unroll
        for (int g = 0; g < GM; ++g) fa[0][g] = frag_ok ? *reinterpret_cast<const float4 *>(as + 32 * g) : float4{};
#pragma unroll
        for (int h = 0; h < GN; ++h) fb[0][h] = frag_ok ? *reinterpret_cast<const float4 *>(bs + 16 * h) : float4{};
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const int cur = kk & 1;
            if (kk + 1 < BK) {
                const int nxt = cur ^ 1;
#pragma unroll
                for (int g = 0; g < GM; ++g)
                    fa[nxt][g] = frag_ok ? *reinterpret_cast<const float4 *>(as + (kk + 1) * A_LD + 32 * g) : float4{};
#pragma unroll
                for (int h = 0; h < GN; ++h)
                    fb[nxt][h] = frag_ok ? *reinterpret_cast<const float4 *>(bs + (kk + 1) * B_LD + 16 * h) : float4{};
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
            // the outer product as packed pairs of neighbouring columns:
            // TM * TN / 2 instructions instead of TM * TN (per output still
            // one rounded fused multiply-add per k, in increasing k)
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; j += 2) fma2(acc[i][j], acc[i][j + 1], a[i], a[i], b[j], b[j + 1]);
        }
    }
    cp_async_wait<0>();

    // ---- epilogue
    const float alpha = p.alpha, beta = p.beta;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + a_off + 32 * (i / 4) + (i % 4);
        if (row >= p.m) continue;
        float *crow = Cb + (long long)row * p.ldc;
#pragma unroll
        for (int h = 0; h < GN; ++h) {
            const int col = n0 + b_off + 16 * h;
            const float *v = &acc[i][4 * h];
            if (p.c_vec && col + 3 < p.n) {
                if (!SG_IN(in_matrix(crow + col, 4, Cb, p.ldc, p.m, p.n))) continue;
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
                    if (col + q < p.n && SG_IN(in_matrix(crow + col + q, 1, Cb, p.ldc, p.m, p.n))) {
                        crow[col + q] = beta != 0.f ? fmaf(alpha, v[q], beta * crow[col + q]) : alpha * v[q];
                    }
                }
            }
        }
    }
}

// The configurations the library launches, both 128 x 128 tiles at two
// CTAs per SM: 8 x 8 per thread (256 threads) for problems of less than
// one wave of 2 CTAs per SM, and 8 x 16 per thread (128 threads, up to 256
// registers each) otherwise -- 6 LDS.128 per 128 FMA instead of 4 per 64,
// and the other CTA's warps cover a CTA's barrier and slab-boundary
// bubbles.  Measured (one GB300, interleaved): 8192^3 64.4 against 60.4
// TFLOPS, 4096^3 60.7 against 57.7, 2048^3 (0.84 waves) 48.0 against 48.5;
// a 128 x 256 tile of 8 x 16 at one CTA per SM ran 62.2, 54.2 and 52.8.
using Default = Config<128, 128, 32, 3, 8, 8, 2>;
using Deep = Config<128, 128, 32, 3, 8, 16, 2>;

// Operand loaders of a configuration by storage: k contiguous ->
// ScatterLoader; rows contiguous -> DirectLoader with 16-byte (rows 16-byte
// aligned) or 4-byte copies.
template <class Cfg>
struct Loaders {
    using AScatter = ScatterLoader<Cfg::BM, Cfg::BK, Cfg::THREADS>;
    using AVec = DirectLoader<Cfg::BM, Cfg::BK, Cfg::THREADS, true>;
    using AScalar = DirectLoader<Cfg::BM, Cfg::BK, Cfg::THREADS, false>;
    using BScatter = ScatterLoader<Cfg::BN, Cfg::BK, Cfg::THREADS>;
    using BVec = DirectLoader<Cfg::BN, Cfg::BK, Cfg::THREADS, true>;
    using BScalar = DirectLoader<Cfg::BN, Cfg::BK, Cfg::THREADS, false>;
};

// Dynamic shared memory of the instance for loader kinds akind / bkind
// (0 scatter, 1 direct 16-byte, 2 direct 4-byte).
template <class Cfg>
constexpr int smem_bytes(int akind, int bkind) {
    using L = Loaders<Cfg>;
    return akind == 0   ? (bkind == 0   ? Layout<Cfg, typename L::AScatter, typename L::BScatter>::SMEM_BYTES
                           : bkind == 1 ? Layout<Cfg, typename L::AScatter, typename L::BVec>::SMEM_BYTES
                                        : Layout<Cfg, typename L::AScatter, typename L::BScalar>::SMEM_BYTES)
           : akind == 1 ? (bkind == 0   ? Layout<Cfg, typename L::AVec, typename L::BScatter>::SMEM_BYTES
                           : bkind == 1 ? Layout<Cfg, typename L::AVec, typename L::BVec>::SMEM_BYTES
                                        : Layout<Cfg, typename L::AVec, typename L::BScalar>::SMEM_BYTES)
                        : (bkind == 0   ? Layout<Cfg, typename L::AScalar, typename L::BScatter>::SMEM_BYTES
                           : bkind == 1 ? Layout<Cfg, typename L::AScalar, typename L::BVec>::SMEM_BYTES
                                        : Layout<Cfg, typename L::AScalar, typename L::BScalar>::SMEM_BYTES);
}

}  // namespace ffma

// C = beta * C over an m x n window (beta == 0 writes zeros without reading);
// blockIdx.y selects the problem of a strided batch (C + y*stride_c).
static __global__ void scale_c_kernel(float *C, long long ldc, int m, int n, float beta, long long stride_c) {
    C += blockIdx.y * stride_c;
    const long long total = (long long)m * n;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long i = idx / n, j = idx - i * n;
        float *c = C + i * ldc + j;
        if (SG_IN(in_matrix(c, 1, C, ldc, m, n))) *c = beta != 0.f ? beta * *c : 0.f;
    }
}

}  // namespace sgemm_gb300
