// 3xTF32 split-precision SGEMM on the sm_103a tensor cores (tcgen05, TMEM).
//
// Not on the pages (they only describe CUDA-core FFMA kernels); this is the
// tensor-core path for the same C = alpha*A*B + beta*C.  Each FP32 operand
// x is split into two TF32 numbers, hi and lo = tf32(x - hi), and
//     a*b ~= a_hi*b_hi + a_hi*b_lo + a_lo*b_hi,
// every product exact in the tensor core and accumulated in FP32 in tensor
// memory.  With the split pass's round-to-nearest hi, |a_lo| <= 2^-11 |a|
// and the dropped a_lo*b_lo term plus the rounding of the lo parts stay
// below ~3 * 2^-22 |a||b| per product; with an operand read as stored (hi =
// x with its low 13 mantissa bits dropped, how the MMA reads FP32), below
// ~2^-19 |a||b|: far inside the FP32 acceptance bound
// |C - r| <= 1e-5 * sum_t |A_it||B_tj| + 1e-6 |beta C0|.
//
// One launch per call, or two:
//  0. (only for an operand TMA cannot read as stored -- rows not 16 bytes
//     apart, a misaligned base -- or, for B, problems above 2^31
//     multiply-adds) the split pass, split_pair_kernel: the operand becomes
//     hi, lo row-major with k contiguous (row pitch ka = k rounded up to 4);
//     a k-major operand (B stored k x n) is transposed through a 32 x 64
//     shared tile padded to 65 columns;
//  1. the GEMM kernel, 12 warps, one CTA per 128 x BN tile of C (BN = 256,
//     or 128 for narrow or few-tile problems; the rest says 256):
//     warp 0 lane 0: TMA producer -- per 16-deep k slab, the MMA's 128-row
//       operand X and its 256-row operand Y into a 4-stage ring (48 KB per
//       stage: [X hi | X lo | Y hi | Y lo]), completing on the slot's "full"
//       mbarrier; an operand read as stored is one raw box (K-major: 64-byte
//       rows, 64-byte swizzle) or 32-row boxes (MN-major: 128-byte swizzle
//       of 32-byte atoms) into its hi slot; a split operand is two boxes;
//       a slot is refilled after the MMA commit for it arrives on its
//       "empty" mbarrier;
//     warps 10, 11: splitters -- for each operand read as stored, lo =
//       tf32(x - trunc(x)) of the raw slab into its lo slot (elementwise, so
//       the swizzle does not matter), a proxy fence, and an arrival on the
//       slot's "converted" barrier of that operand;
//     warp 1: allocates 512 TMEM columns (two 128 x 256 FP32 accumulators);
//       lane 0 issues, per 8-deep k step, the three tcgen05.mma kind::tf32
//       (128 x 256 x 8): hi x hi as soon as the slab lands, each product
//       with a lo part of a raw operand once it is converted; it commits
//       each slab back to its "empty" barrier;
//     warps 2-9: FP32 accumulation on the CUDA cores.  The tensor core's
//       own FP32 accumulation is not round-to-nearest: its error is biased
//       and grows with the number of accumulation steps (measured: 0.31 of
//       the bound at k = 8192 on N(0,1) data, and it would exceed the bound on
//       non-negative data).  So the MMA accumulates only KC = 128 k at a
//       time, alternating between the two TMEM accumulators; for each such
//       chunk these warps load their part (32 lanes = rows, 128 columns)
//       with tcgen05.ld and add it into FP32 registers with round-to-nearest
//       adds, then release the TMEM buffer.  After the last chunk they write
//       alpha*acc + beta*C for rows < m, columns < n (C not read when
//       beta == 0), 32 columns of each warp's 32 rows at a time through the
//       warp's 4 KB staging buffer in shared memory, so that every store
//       covers 4 rows x 128 contiguous bytes.
//     Split-K for problems with too few tiles to fill the GPU: the grid is
//     launched in clusters of S CTAs (S <= 8) that share one tile, CTA r
//     taking k slabs [r*KT/S, (r+1)*KT/S).  Each parks its FP32 partial
//     tile in its own shared memory; after a cluster barrier CTA r sums
//     rows [r*128/S, (r+1)*128/S) over all S partials in rank order through
//     distributed shared memory (ld.shared::cluster) and writes them to C,
//     then a second cluster barrier keeps every partial alive until read.
//     The reduction order is fixed, so results do not depend on timing.
//     Narrow problems (n <= 128, TRANS): a 128 x 128 x 8 MMA takes about
//     as long as a 128 x 256 x 8 one, so these compute tiles of
//     C^T = B^T A^T instead -- the MMA's 128-row operand is B^T (the n side),
//     its 256-row operand is A (256 rows of C per tile) -- and the
//     accumulator warps store C^T's rows as columns of C (each warp's 32
//     lanes are 32 consecutive columns: 128-byte stores).
//     Stream-K (Params): persistent CTAs that take whole tiles for the full
//     waves and share the last wave's tiles out by slabs, a shared tile
//     being finished by the last of its CTAs from partials in a workspace.
//     CTA pairs (Pair config, cta_group::2): two CTAs of a cluster compute a
//     256 x 256 tile with M = 256 MMAs issued by the even CTA; each stages
//     and splits its 128 rows of A and of B (7 stages of 32 KB; C staged in
//     the ring once the tile's last slab is done).
//     After a split pass, a GEMM that runs in one wave is launched as its
//     programmatic dependent: it sets up while the split finishes, and its
//     producer waits for it before the first load.
//     TMA zero-fills rows past m, columns past n and k past the end, so the
//     MMA never sees an index test.  Every mbarrier wait is bounded (2 s):
//     a wait that runs out records a code in the library status word,
//     stops issuing, lets issued copies and MMAs complete (bounded), skips
//     the stores and frees TMEM before the CTA exits.
#pragma once
#include <cuda.h>

#include <cstdint>

#include "ptx.cuh"
#include "raster.cuh"
#include "tcgen05.cuh"

namespace sgemm_gb300 {
namespace tf32x3 {

constexpr int BM = 128;
constexpr int BK = 16;   // 64-byte rows
constexpr int UMMA_K = 8;
constexpr int KC = 128;                                   // k per tensor-core accumulation chunk
constexpr int CHUNK_STAGES = KC / BK;
constexpr int A_TILE = BM * BK * 4;                       // 8 KB
constexpr int ACC_WARPS = 8;
constexpr int ACC_THREADS = 32 * ACC_WARPS;
constexpr int CONV_WARPS = 2;                             // splitters of raw operands
constexpr int CONV_THREADS = 32 * CONV_WARPS;
// producer warp, MMA warp, 8 accumulator warps, 2 splitter warps: three
// warps per sub-partition, a cap of 168 registers per thread
constexpr int THREADS = 64 + ACC_THREADS + CONV_THREADS;
constexpr int BAR_REGION = 512;
static_assert(BK * 4 == 64, "one 64-byte swizzle row per operand row");
static_assert(KC % BK == 0, "chunks are whole slabs");

// Tile width BN (256, or 128 for narrow / few-tile problems) and ring depth.
// PAIR: a CTA pair (cta_group::2) computes a 256 x BN tile with one MMA of
// M = 256; each CTA holds 128 rows of the MMA's A operand and BN / 2 rows of
// its B operand, and receives 128 rows x BN columns of D.
template <int BN_, int STAGES_, bool PAIR_ = false>
struct Config {
    static constexpr int BN = BN_, STAGES = STAGES_;
    static constexpr bool PAIR = PAIR_;
    static constexpr int Y_ROWS = PAIR ? BN / 2 : BN;             // rows of the MMA's B operand in this CTA
    static constexpr int B_TILE = Y_ROWS * BK * 4;
    static constexpr int STAGE_BYTES = 2 * A_TILE + 2 * B_TILE;   // A_hi, A_lo, B_hi, B_lo
    static constexpr int TMEM_COLS = 2 * BN;                      // two accumulators
    static constexpr int COLS_PER_THREAD = BN / 2;                // two warps per 32-lane group
    // C's staging blocks (a 32 x 32 block per accumulator warp, 32 KB): in
    // their own region, or -- for CTA pairs, which never run stream-K, so a
    // CTA stores its one tile only after its last slab -- at the start of
    // the then idle stage ring, which leaves room for a seventh stage
    static constexpr bool EPI_IN_RING = PAIR;
    static constexpr int EPI_BYTES = EPI_IN_RING ? 0 : ACC_WARPS * 32 * 32 * 4;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_REGION + EPI_BYTES;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "power-of-two TMEM allocation");
    static_assert(COLS_PER_THREAD % 16 == 0, "accumulator warps load 16 columns at a time");
};
using Wide = Config<256, 4>;     // 48 KB stages
using Narrow = Config<128, 6>;   // 32 KB stages
using Pair = Config<256, 7, true>;   // 32 KB stages per CTA, 256 x 256 tiles per CTA pair

constexpr int kStatusProducer = 0x201;
constexpr int kStatusMma = 0x202;
constexpr int kStatusAccumulate = 0x203;
constexpr int kStatusDrain = 0x204;
constexpr int kStatusMmaBuffer = 0x205;
constexpr int kStatusSplit = 0x206;

struct Params {
    int m, n, k;
    float alpha, beta;
    float *C;
    long long ldc;
    int tiles_m, tiles_n, group_m;
    // strided batch: problem blockIdx.y writes C + y*stride_c and reads its
    // operands at TMA coordinate z = y (x_z, y_z set: the operand's tensor
    // map has a batch dimension) or z = 0 (one operand shared by the batch)
    long long stride_c;
    int x_z, y_z;
    // where each MMA operand comes from (kPreSplit, kRaw or kPhased, see the
    // kernel); kPhased: bits 2j..2j+1 of x_shift = row phase j's shift
    int x_src, y_src;
    int x_shift;
    // C rows 16-byte aligned (ldc % 4 == 0, C 16-byte aligned): float4 access
    int c_vec;
    // stream-K (sk_ctas > 0, grid = G = sk_ctas persistent CTAs, one
    // problem): with tiles = W G + R, CTA g first takes whole tiles g,
    // g + G, ..., g + (W - 1) G (the full waves, in raster order, so CTAs
    // running at the same time share operand panels in L2), then slabs
    // [T g / G, T (g + 1) / G) of the sequence "tile W G slabs 0..KT-1,
    // tile W G + 1 slabs 0..KT-1, ..." of the R remaining tiles (T = R KT).
    // A CTA that holds only part of a tile writes its partial sums to its
    // slot of sk_ws (2 x BM x BN floats per CTA: slot 0 for the tile its run
    // starts in, slot 1 for the one it ends in) and counts itself in
    // sk_cnt[tile] (zeroed before the launch); the last of a tile's CTAs
    // adds all partials in k order and writes the tile.
    // sk_ctas < 0: persistent whole tiles -- G = -sk_ctas CTAs, CTA g takes
    // tiles g, g + G, g + 2G, ... (a tile's epilogue overlaps the next
    // tile's first chunks: the TMEM buffers alternate across tiles).
    // sk_parts >= 2 (stream-K, R S <= G): the R remaining tiles are cut
    // into S equal k ranges instead, part j of tile W G + i going to CTA
    // i S + j, so that the CTAs of a tile row (column) read the same k
    // range of its A (B) panel at the same time and share it in L2.
    int sk_ctas;
    int sk_parts;
    float *sk_ws;
    int *sk_cnt;
};
// (a parameter block above 128 bytes measurably raised the GEMM kernel's
// register spills)
static_assert(sizeof(Params) <= 128, "kernel parameter block");

// Segment `si` of the work of CTA blockIdx.x -- one tile and a range
// [k0, k0 + nk) of its kt_all slabs; false past the last.  Stream-K over
// sk_ctas > 0 CTAs (see Params): the whole tiles blockIdx.x + w G first, then
// the CTA's run of the remaining tiles' slab sequence cut at tile
// boundaries, or (sk_parts >= 2) its one k part of one remaining tile.
// Persistent whole tiles (sk_ctas < 0): tiles blockIdx.x + w G.  Otherwise one
// segment of tile blockIdx.x / ctas_per_tile (nsplit for a split-K cluster,
// 2 for a CTA pair, else 1): split-K cluster rank `rank`'s share of its
// slabs (possibly empty), or all of them.  Recomputed on demand so that no
// role keeps iteration state next to its accumulators.
__device__ __forceinline__ bool cta_segment(int sk_ctas, int kt_all, int tiles, uint32_t nsplit, uint32_t rank,
                                            int si, int &tile, int &k0, int &nk, int ctas_per_tile, int sk_parts) {
    long long it0, it1;
    if (sk_ctas != 0) {
        // rounds of whole tiles (all of them when persistent)
        const int G = sk_ctas < 0 ? -sk_ctas : sk_ctas;
        const int whole = sk_ctas < 0 ? (tiles + G - 1) / G : tiles / G;
        if (si < whole) {
            tile = (int)blockIdx.x + si * G;
            k0 = 0;
            nk = kt_all;
            return tile < tiles;
        }
        if (sk_ctas < 0) return false;
        si -= whole;
        if (sk_parts >= 2) {
            // one k part of one remaining tile per CTA
            const int g = (int)blockIdx.x, first = whole * sk_ctas;
            if (si != 0 || g >= (tiles - first) * sk_parts) return false;
            tile = first + g / sk_parts;
            const int j = g % sk_parts;
            k0 = (int)((long long)kt_all * j / sk_parts);
            nk = (int)((long long)kt_all * (j + 1) / sk_parts) - k0;
            return nk > 0;
        }
        const long long base = (long long)whole * sk_ctas * kt_all;
        const long long T = (long long)(tiles - whole * sk_ctas) * kt_all;
        it0 = base + T * blockIdx.x / sk_ctas;
        it1 = base + T * (blockIdx.x + 1) / sk_ctas;
    } else {
        if (si > 0) return false;
        tile = (int)blockIdx.x / ctas_per_tile;
        k0 = (int)((long long)kt_all * rank / nsplit);
        nk = (int)((long long)kt_all * (rank + 1) / nsplit) - k0;
        return true;
    }
    const long long t = it0 / kt_all + si, tb = t * kt_all;
    if (tb >= it1) return false;
    const long long lo = si == 0 ? it0 : tb;
    const long long hi = it1 < tb + kt_all ? it1 : tb + kt_all;
    tile = (int)t;
    k0 = (int)(lo - tb);
    nk = (int)(hi - lo);
    return true;
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// Barrier `id` over `threads` threads that also returns whether any of them
// passed true (every participant gets the same answer).
__device__ __forceinline__ bool named_barrier_or(int id, int threads, bool v) {
    uint32_t out;
    asm volatile(
        "{\n"
        ".reg .pred p, q;\n"
        "setp.ne.u32 q, %1, 0;\n"
        "bar.red.or.pred p, %2, %3, q;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(out)
        : "r"((uint32_t)v), "r"(id), "r"(threads)
        : "memory");
    return out != 0;
}

// ---------------------------------------------------------------- split kernels

__device__ __forceinline__ void split_one(float x, float &h, float &l) {
    h = tc::round_tf32(x);
    l = tc::round_tf32(x - h);
}

// The lo part of x when x itself is the MMA's hi operand: a kind::tf32 MMA
// reads an FP32 operand with its low 13 mantissa bits dropped (measured on
// GB300: every output of x * I equals x truncated to TF32, ties and all), so
// hi = trunc(x); r = x - hi is exact in FP32 and lo = tf32(r), rounded to
// nearest with ties away from zero, with |x - hi - lo| <= 2^-11 |r| <
// 2^-21 |x|.  The rounding is done on the bits: add half of the dropped
// range to the magnitude (|r| < 2^-10 |x| cannot round up to infinity).
// Dropping the low 13 bits afterwards is left to the MMA, which reads them
// that way -- the product is the same as with cvt.rna.tf32 -- so a value
// costs three operations (the conversion instruction measured ~6 % slower
// in the splitter warps at 8192^3).  The result is meant for the MMA only.
__device__ __forceinline__ float lo_of_raw(float x) {
    const float h = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    return __uint_as_float(__float_as_uint(x - h) + 0x1000u);
}

// d0 = a0 - b0, d1 = a1 - b1 as one packed instruction (sub.rn.f32x2).
__device__ __forceinline__ void sub2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
    asm("{\n"
        ".reg .b64 ra, rb, rd;\n"
        "mov.b64 ra, {%2, %3};\n"
        "mov.b64 rb, {%4, %5};\n"
        "sub.rn.f32x2 rd, ra, rb;\n"
        "mov.b64 {%0, %1}, rd;\n"
        "}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// lo_of_raw of four values, the subtractions as two packed instructions.
__device__ __forceinline__ float4 lo4_of_raw(float4 x) {
    const float hx = __uint_as_float(__float_as_uint(x.x) & 0xFFFFE000u);
    const float hy = __uint_as_float(__float_as_uint(x.y) & 0xFFFFE000u);
    const float hz = __uint_as_float(__float_as_uint(x.z) & 0xFFFFE000u);
    const float hw = __uint_as_float(__float_as_uint(x.w) & 0xFFFFE000u);
    float4 r;
    sub2(r.x, r.y, x.x, x.y, hx, hy);
    sub2(r.z, r.w, x.z, x.w, hz, hw);
    return make_float4(__uint_as_float(__float_as_uint(r.x) + 0x1000u), __uint_as_float(__float_as_uint(r.y) + 0x1000u),
                       __uint_as_float(__float_as_uint(r.z) + 0x1000u), __uint_as_float(__float_as_uint(r.w) + 0x1000u));
}

// A (m x k, row pitch lda) -> hi, lo (m x ka, row pitch ka).  VEC: A and
// lda 16-byte aligned, so every row is read as float4 except a k % 4 tail
// (read element by element: the bytes past k may lie outside A).
// The work of block (bx, by) of a gx x gy grid, on problem bz of a strided
// batch (split_a_kernel runs it on its own grid, split_pair_kernel on part
// of a shared one).
template <bool VEC>
__device__ __forceinline__ void split_rows(const float *__restrict__ A, long long lda, int m, int k,
                                           float *__restrict__ hi, float *__restrict__ lo, int ka,
                                           long long src_batch, long long dst_batch, int bx, int by, int bz, int gx,
                                           int gy) {
    A += bz * src_batch;
    hi += bz * dst_batch;
    lo += bz * dst_batch;
    const int full4 = VEC ? k / 4 : 0;               // float4 chunks entirely inside the row
    const int scal0 = 4 * full4;                      // first element done one at a time
    const int stride = gx * (int)blockDim.x;
    for (int row = by; row < m; row += gy) {
        const float *src = A + (long long)row * lda;
        float *h = hi + (long long)row * ka;
        float *l = lo + (long long)row * ka;
        for (int c = bx * (int)blockDim.x + (int)threadIdx.x; c < full4; c += stride) {
            if (!SG_IN(in_matrix(src + 4 * c, 4, A, lda, m, k) && in_matrix(h + 4 * c, 4, hi, ka, m, ka) &&
                       in_matrix(l + 4 * c, 4, lo, ka, m, ka)))
                continue;
            const float4 x = __ldg(reinterpret_cast<const float4 *>(src) + c);
            float4 xh, xl;
            split_one(x.x, xh.x, xl.x);
            split_one(x.y, xh.y, xl.y);
            split_one(x.z, xh.z, xl.z);
            split_one(x.w, xh.w, xl.w);
            reinterpret_cast<float4 *>(h)[c] = xh;
            reinterpret_cast<float4 *>(l)[c] = xl;
        }
        for (int t = scal0 + bx * (int)blockDim.x + (int)threadIdx.x; t < k; t += stride) {
            if (!SG_IN(in_matrix(src + t, 1, A, lda, m, k) && in_matrix(h + t, 1, hi, ka, m, ka) &&
                       in_matrix(l + t, 1, lo, ka, m, ka)))
                continue;
            float xh, xl;
            split_one(__ldg(src + t), xh, xl);
            h[t] = xh;
            l[t] = xl;
        }
    }
}

template <bool VEC>
__global__ void __launch_bounds__(256) split_a_kernel(const float *__restrict__ A, long long lda, int m, int k,
                                                      float *__restrict__ hi, float *__restrict__ lo, int ka,
                                                      long long src_batch, long long dst_batch) {
    griddep_launch_dependents();   // the GEMM may start its set-up meanwhile
    split_rows<VEC>(A, lda, m, k, hi, lo, ka, src_batch, dst_batch, (int)blockIdx.x, (int)blockIdx.y,
                    (int)blockIdx.z, (int)gridDim.x, (int)gridDim.y);
}

// One split pass of a GEMM call: a k-contiguous operand is split row by row
// (split_rows; kind 1 with float4 loads when its rows are 16-byte aligned);
// a k-major one (B, k x n, row pitch ld) becomes hi, lo of its transpose
// (n x ka, row pitch ka) through a 32 (k) x 64 (n) shared tile padded to 65
// columns: reads of B and writes of B^T are both 128-byte coalesced per
// warp, and the column reads of the tile hit 32 different banks.  gx x gy
// blocks per problem.
struct SplitJob {
    const float *src;
    long long ld;
    int rows, cols;   // rows x k (kinds 0, 1), or k x n (transpose)
    float *hi, *lo;
    int ka;
    long long src_batch, dst_batch;
    int gx, gy;
    int kind;         // 0: split_rows, 1: split_rows with float4 loads, 2: transpose
};

// The split passes of a GEMM call in one launch (one launch gap fewer before
// the GEMM when both operands are split): blocks [0, j0.gx * j0.gy) of each
// batch slice run job j0, the rest job j1 (none when j1.gx = 0).  The branch
// is uniform per block.  The transpose is written out here rather than in a
// device function: that form measured ~19 % slower on GB300 (B of 8192 x
// 8192: 209.6 against 176.8 us).
static __global__ void __launch_bounds__(256) split_pair_kernel(SplitJob j0, SplitJob j1) {
    griddep_launch_dependents();   // the GEMM may start its set-up meanwhile
    const int n0 = j0.gx * j0.gy;
    const bool first = (int)blockIdx.x < n0;
    const SplitJob j = first ? j0 : j1;
    const int b = first ? (int)blockIdx.x : (int)blockIdx.x - n0;
    const int bx = b % j.gx, by = b / j.gx, bz = (int)blockIdx.z;
    if (j.kind != 2) {
        if (j.kind == 1)
            split_rows<true>(j.src, j.ld, j.rows, j.cols, j.hi, j.lo, j.ka, j.src_batch, j.dst_batch, bx, by, bz,
                             j.gx, j.gy);
        else
            split_rows<false>(j.src, j.ld, j.rows, j.cols, j.hi, j.lo, j.ka, j.src_batch, j.dst_batch, bx, by, bz,
                              j.gx, j.gy);
        return;
    }
    __shared__ float tile[32][65];
    const float *B = j.src + bz * j.src_batch;
    float *hi = j.hi + bz * j.dst_batch, *lo = j.lo + bz * j.dst_batch;
    const int k = j.rows, n = j.cols, ka = j.ka;
    const long long ldb = j.ld;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
    for (int t0 = by * 32; t0 < k; t0 += j.gy * 32) {
        for (int j0_ = bx * 64; j0_ < n; j0_ += j.gx * 64) {
#pragma unroll
            for (int r = ty; r < 32; r += 8) {
                const int t = t0 + r;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int jj = j0_ + 32 * q + tx;
                    const bool in = t < k && jj < n && SG_IN(in_matrix(B + (long long)t * ldb + jj, 1, B, ldb, k, n));
                    tile[r][32 * q + tx] = in ? __ldg(B + (long long)t * ldb + jj) : 0.f;
                }
            }
            __syncthreads();
#pragma unroll
            for (int r = ty; r < 64; r += 8) {
                const int jj = j0_ + r, t = t0 + tx;
                if (jj < n && t < k && SG_IN(in_matrix(hi + (long long)jj * ka + t, 1, hi, ka, n, ka))) {
                    float xh, xl;
                    split_one(tile[tx][r], xh, xl);
                    hi[(long long)jj * ka + t] = xh;
                    lo[(long long)jj * ka + t] = xl;
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------- GEMM kernel

// The MMA's two operands: X, its 128-row A operand, and Y, its BN-row B
// operand.  Untransposed tiles: X = rows of A (m side), Y = columns of B
// (n side).  TRANS tiles: X = columns of B, Y = rows of A.
//
// Each operand reaches a stage slot in one of these ways (Params::x_src,
// y_src; kPhased below for X only):
//   kPreSplit: its hi and lo parts were written by the split pass (K-major,
//     row pitch ka) and TMA loads both;
//   kRaw: TMA loads the operand as the caller stored it into the hi slot --
//     K-major (rows of consecutive k: A stored m x k, B stored n x k) in
//     64-byte rows with the 64-byte swizzle, or MN-major (X_MN / Y_MN: rows
//     of consecutive m or n: A stored k x m, B stored k x n) in boxes of
//     32 rows x 16 k with the 128-byte swizzle of 32-byte atoms.  The MMA reads that FP32 slab as
//     its hi part (a kind::tf32 MMA drops the low 13 mantissa bits), and the
//     two splitter warps (10, 11) write lo = tf32(x - hi) into the lo slot
//     at the same (swizzled) position, make the writes visible to the tensor
//     core's proxy and arrive on the slot's "converted" barrier of that
//     operand.  The MMA issuer sends hi x hi as soon as the slab lands and
//     waits for an operand's lo only before the product that reads it.
// Error of a raw operand: hi = trunc(x), |x - hi - lo| < 2^-21 |x| and
// |lo| < 2^-10 |x| (against 2^-22 and 2^-11 for the split pass's
// round-to-nearest hi), so each product stays within ~2^-19 |a b| of exact
// even with both operands raw, far inside the FP32 acceptance bound.
constexpr int kPreSplit = 0;
constexpr int kRaw = 1;
// kPhased: X (K-major A on untransposed single-CTA tiles) whose rows TMA
// cannot read as one tensor -- rows not 16 bytes apart, or a misaligned
// base.  Every fourth row is, though: the rows 4i + j of row phase j
// (j = 0..3) are 4 * lda floats apart, a multiple of 16 bytes, so each
// phase is a tensor of its own, based at its first row rounded down to 16
// bytes, where each row starts sh_j (0..3) floats into its own row of the
// view.  TMA loads the four phases' 32-row boxes of PHASE_COLS = 20 columns
// (16 k and the shift) into a staging area over the X hi and lo slots; the
// splitter warps read each row's 16 values from sh_j on, then write hi
// (the value as stored) and lo into the swizzled slots, where the MMA takes
// them like a raw operand's -- hi x hi too only after that.
constexpr int kPhased = 2;
constexpr int PHASE_COLS = 20;
constexpr int PHASE_BOX = (BM / 4) * PHASE_COLS * 4;   // one phase's 32 rows, bytes
constexpr int PHASE_BYTES = 4 * PHASE_BOX;
static_assert(PHASE_BYTES <= 2 * A_TILE, "staging fits over the X hi and lo slots");

// Loads one operand's part of a slab: `rows` rows starting at row0 and 16 k
// starting at kx, of problem z.  K-major: one box (16 k x rows); MN-major:
// rows / 32 boxes (32 rows x 16 k, 2 KB each) side by side.
template <bool MN, int ROWS>
__device__ __forceinline__ void load_operand(uint32_t hi_slot, uint32_t lo_slot, const CUtensorMap *map_hi,
                                             const CUtensorMap *map_lo, bool raw, int row0, int kx, int z,
                                             uint32_t bar) {
    if constexpr (MN) {
#pragma unroll
        for (int j = 0; j < ROWS / 32; ++j) tma_load_3d(hi_slot + j * 2048, map_hi, row0 + 32 * j, kx, z, bar);
    } else {
        tma_load_3d(hi_slot, map_hi, kx, row0, z, bar);
        if (!raw) tma_load_3d(lo_slot, map_lo, kx, row0, z, bar);
    }
}

// Descriptor of k step kk (8 values) of an operand slot.
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t slot, int kk) {
    if constexpr (MN)
        return tc::desc_mnmajor_sw128_32b(slot + (uint32_t)kk * 1024u);
    else
        return tc::desc_kmajor_sw64(slot + (uint32_t)kk * (UMMA_K * 4));
}

// lo = tf32(x - trunc(x)) of every value of a raw slot, in place order,
// by `cw` threads (this one is `ct`), eight 16-byte loads in flight each.
template <int BYTES, int CW>
__device__ __forceinline__ void split_slot_lo(const uint8_t *raw_slot, uint8_t *lo_slot, int ct) {
    constexpr int PER = BYTES / 16 / CW;   // float4 per thread
    static_assert(BYTES % (16 * CW) == 0, "whole float4s per thread");
    const float4 *raw = reinterpret_cast<const float4 *>(raw_slot);
    float4 *lo = reinterpret_cast<float4 *>(lo_slot);
    constexpr int G = PER < 8 ? PER : 8;
#pragma unroll
    for (int j0 = 0; j0 < PER; j0 += G) {
        float4 x[G];
#pragma unroll
        for (int j = 0; j < G; ++j) x[j] = raw[ct + (j0 + j) * CW];
#pragma unroll
        for (int j = 0; j < G; ++j)
            lo[ct + (j0 + j) * CW] = lo4_of_raw(x[j]);
    }
}

// Both lo parts of a slab at once: every thread's 16-byte loads of X and Y
// in flight together, then the conversions and the stores.
template <int XBYTES, int YBYTES, int CW>
__device__ __forceinline__ void split_slots_lo(const uint8_t *x_raw, uint8_t *x_lo, const uint8_t *y_raw,
                                               uint8_t *y_lo, int ct) {
    constexpr int PX = XBYTES / 16 / CW, PY = YBYTES / 16 / CW;
    static_assert(XBYTES % (16 * CW) == 0 && YBYTES % (16 * CW) == 0, "whole float4s per thread");
    const float4 *xr = reinterpret_cast<const float4 *>(x_raw), *yr = reinterpret_cast<const float4 *>(y_raw);
    float4 *xl = reinterpret_cast<float4 *>(x_lo), *yl = reinterpret_cast<float4 *>(y_lo);
    float4 v[PX + PY];
#pragma unroll
    for (int j = 0; j < PX; ++j) v[j] = xr[ct + j * CW];
#pragma unroll
    for (int j = 0; j < PY; ++j) v[PX + j] = yr[ct + j * CW];
#pragma unroll
    for (int j = 0; j < PX + PY; ++j) v[j] = lo4_of_raw(v[j]);
#pragma unroll
    for (int j = 0; j < PX; ++j) xl[ct + j * CW] = v[j];
#pragma unroll
    for (int j = 0; j < PY; ++j) yl[ct + j * CW] = v[PX + j];
}

// A phased X slab (kPhased): the four phases' staged boxes at hi_slot
// (phase j's 32 rows of PHASE_COLS floats at j * PHASE_BOX; its rows start
// sh_j = bits 2j..2j+1 of `shifts` floats in) -> hi (the value as stored)
// and lo, K-major in the 64-byte swizzle (16-byte chunk q of row r at chunk
// q ^ ((r >> 1) & 3)).  The staging lies over both slots, so the CW threads
// (this one is ct) read all of their values first and meet at a barrier
// (named barrier 2 for two warps) before writing.  A warp reads one
// 16-byte chunk q of rows 4i + j and 4(i + 4) + j (j = 0..3) per lane:
// its 32 loads fall in 32 distinct banks when the four shifts differ (lda
// odd).
template <int CW>
__device__ __forceinline__ void split_phased(uint8_t *hi_slot, uint8_t *lo_slot, uint32_t shifts, int ct) {
    constexpr int UNITS = 16 / (CW / 32);   // warp-wide reads of 32 chunks per thread
    const int lane = ct & 31, q = lane & 3, j = (lane >> 2) & 3;
    const float *stg = reinterpret_cast<const float *>(hi_slot) + j * (PHASE_BOX / 4) + ((shifts >> (2 * j)) & 3) + 4 * q;
    float4 v[UNITS];
#pragma unroll
    for (int t = 0; t < UNITS; ++t) {
        const int u = (ct >> 5) + (CW / 32) * t;
        const int i = (u & 3) + 8 * (u >> 2) + 4 * (lane >> 4);
        const float *x = stg + i * PHASE_COLS;
        v[t] = SG_IN(x + 4 <= reinterpret_cast<const float *>(hi_slot) + PHASE_BYTES / 4) ? make_float4(x[0], x[1], x[2], x[3])
                                                                                       : float4{};
    }
    if constexpr (CW == 32)
        __syncwarp();
    else
        named_barrier_sync(2, CW);
#pragma unroll
    for (int t = 0; t < UNITS; ++t) {
        const int u = (ct >> 5) + (CW / 32) * t;
        const int r = 4 * ((u & 3) + 8 * (u >> 2) + 4 * (lane >> 4)) + j;
        const int off = r * 64 + ((q ^ ((r >> 1) & 3)) << 4);
        if (!SG_IN(off + 16 <= A_TILE)) continue;
        *reinterpret_cast<float4 *>(hi_slot + off) = v[t];
        *reinterpret_cast<float4 *>(lo_slot + off) = lo4_of_raw(v[t]);
    }
}

// X_PH: X is read in row phases (kPhased); a separate instantiation, so
// that the others carry none of its code (which measured ~3 % at 8192^3).
template <class Cfg, bool TRANS = false, bool X_MN = false, bool Y_MN = false, bool X_PH = false>
__global__ void __launch_bounds__(THREADS, 1)
    tf32x3_gemm_kernel(const __grid_constant__ CUtensorMap tmXhi, const __grid_constant__ CUtensorMap tmXlo,
                       const __grid_constant__ CUtensorMap tmYhi, const __grid_constant__ CUtensorMap tmYlo,
                       const __grid_constant__ CUtensorMap tmX2, const __grid_constant__ CUtensorMap tmX3,
                       const Params p) {
    constexpr int BN = Cfg::BN, STAGES = Cfg::STAGES, Y_TILE = Cfg::B_TILE, STAGE_BYTES = Cfg::STAGE_BYTES;
    constexpr int X_TILE = A_TILE;
    constexpr bool PAIR = Cfg::PAIR;
    constexpr int Y_ROWS = Cfg::Y_ROWS;
    static_assert(!PAIR || !TRANS, "CTA pairs compute untransposed tiles");
    constexpr int TMEM_COLS = Cfg::TMEM_COLS, COLS_PER_THREAD = Cfg::COLS_PER_THREAD;
    constexpr int PART_PITCH = BN + 4;   // floats per row of a parked split-K partial tile
    constexpr int NTHREADS = THREADS;
    constexpr bool CONV_PER_WARP = BN == 128;   // splitters: one warp per slab (see there)
    static_assert(!PAIR || !CONV_PER_WARP, "PAIR: both splitter warps take every slab (they meet at a barrier)");
    // slots of a stage: [X hi | X lo | Y hi | Y lo]
    constexpr int X_HI = 0, X_LO = X_TILE, Y_HI = 2 * X_TILE, Y_LO = 2 * X_TILE + Y_TILE;
    static_assert(X_LO % 1024 == 0 && Y_HI % 1024 == 0 && Y_LO % 1024 == 0 && STAGE_BYTES % 1024 == 0,
                  "slots on 1 KB boundaries (128-byte swizzle atoms)");
    static_assert(!X_MN || X_TILE == (BM / 32) * 2048, "MN-major X: 32-row boxes of 2 KB");
    static_assert(!Y_MN || Y_TILE == (Y_ROWS / 32) * 2048, "MN-major Y: 32-row boxes of 2 KB");
    static_assert(BM * PART_PITCH * 4 <= STAGES * STAGE_BYTES, "partial tile fits the stage memory");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *const smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t stage0 = smem_u32(smem);
    uint8_t *const bars = smem + STAGES * STAGE_BYTES;
    const uint32_t bar_full = smem_u32(bars);            // [STAGES] TMA landed
    const uint32_t bar_empty = bar_full + 8 * STAGES;    // [STAGES] MMAs done reading the slot
    const uint32_t bar_tfull = bar_empty + 8 * STAGES;   // [2] chunk accumulated in TMEM buffer b
    const uint32_t bar_tempty = bar_tfull + 16;          // [2] TMEM buffer b drained to registers
    const uint32_t bar_done = bar_tempty + 16;           // every MMA issued has completed
    uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(bars + 8 * (2 * STAGES + 5));
    volatile int *const abort_flag = reinterpret_cast<volatile int *>(bars + 8 * (2 * STAGES + 5) + 8);
    volatile int *const sk_last = reinterpret_cast<volatile int *>(bars + 8 * (2 * STAGES + 5) + 12);
    const uint32_t bar_conv_x = bar_done + 24;           // [STAGES] X's lo written (raw X)
    const uint32_t bar_conv_y = bar_conv_x + 8 * STAGES; // [STAGES] Y's lo written (raw Y)
    // PAIR: [STAGES] the peer's slab landed and its lo parts are written
    // (transaction bytes of a 16-byte signal copy the peer sends), and the
    // 16-byte landing / source pad of that copy
    const uint32_t bar_peer = bar_conv_y + 8 * STAGES;
    const uint32_t sig_pad = (bar_peer + 8 * STAGES + 15) & ~15u;
    // [ACC_WARPS][32 rows][8 float4]
    float4 *const epi = reinterpret_cast<float4 *>(Cfg::EPI_IN_RING ? smem : bars + BAR_REGION);
    static_assert(!Cfg::EPI_IN_RING || ACC_WARPS * 32 * 32 * 4 <= STAGES * STAGE_BYTES, "staging fits the ring");
    static_assert(8 * (5 * STAGES + 7) + 32 <= BAR_REGION, "barrier region");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    static_assert(!X_PH || (!TRANS && !X_MN && !PAIR), "row phases: K-major X on untransposed single-CTA tiles");
    constexpr bool x_ph = X_PH;   // X loaded in row phases (p.x_src == kPhased)
    const bool x_raw = p.x_src == kRaw || x_ph, y_raw = p.y_src == kRaw;
    const bool c_vec = p.c_vec != 0;
    // split-K: the CTAs of a cluster share one output tile and take
    // consecutive ranges of its k slabs (a cluster of one without split-K).
    // PAIR: the cluster is the CTA pair, which shares one tile and all of k;
    // its even CTA (the leader) issues the MMAs, and `prank` (0 / 1) picks
    // this CTA's half of the tile's rows and of its B operand
    const uint32_t crank = tc::cluster_ctarank();
    const uint32_t nsplit = PAIR ? 1u : tc::cluster_nctarank(), rank = PAIR ? 0u : crank;
    const uint32_t prank = PAIR ? (crank & 1u) : 0u, leader = crank & ~1u;
    constexpr int CTAS_PER_TILE_PAIR = PAIR ? 2 : 1;
    const int CTAS_PER_TILE = PAIR ? CTAS_PER_TILE_PAIR : (int)nsplit;
    // TRANS: the tile is BN rows of C by BM columns (C^T = B^T A^T: the
    // MMA's 128-row operand is B^T, its BN-row operand is A).  PAIR: 256 x BN
    constexpr int TILE_M = TRANS ? BN : (PAIR ? 2 * BM : BM), TILE_N = TRANS ? BM : BN;
    float *const Cb = p.C + (long long)blockIdx.y * p.stride_c;
    const int KT_ALL = (p.k + BK - 1) / BK;
    const int tiles = p.tiles_m * p.tiles_n;
    // stream-K's CTA count (CTA pairs never run stream-K: a constant 0 lets
    // the compiler drop those paths)
    const int SK_CTAS = PAIR ? 0 : p.sk_ctas;
    const int SK_PARTS = PAIR ? 0 : p.sk_parts;
    const bool sk = SK_CTAS > 0;
    // this CTA's work: whole tiles of the full waves and a share of the
    // remaining tiles' slabs (stream-K), a consecutive range of one tile's
    // slabs (split-K cluster rank `rank`), or one whole tile
    // (cta_segment above walks it)
    auto tile_origin = [&](int t, int &m0, int &n0) {
        int tm, tn;
        raster_tile(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        m0 = tm * TILE_M;
        n0 = tn * TILE_N;
    };
    // the split-K cluster's tile (its reduction below writes it)
    int cl_m0 = 0, cl_n0 = 0;
    if (nsplit > 1) tile_origin((int)(blockIdx.x / nsplit), cl_m0, cl_n0);
    // PAIR: one arrival at barrier `bar` of the pair's leader -- a plain
    // arrival in the leader itself, a cluster-scope release from its peer
    auto arrive_leader = [&](uint32_t bar) {
        if (prank == 0)
            mbar_arrive(bar);
        else
            mbar_arrive_cluster(tc::map_shared_rank(bar, leader));
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        // PAIR: each CTA's accumulator warps arrive once at the leader's
        // "drained" barrier (an elected thread after their named barrier);
        // the per-slab signal from the peer is the transaction bytes of its
        // signal copy, expected by the leader's MMA thread (one arrival)
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + 8 * b, 1);
            mbar_init(bar_tempty + 8 * b, PAIR ? 2 : ACC_THREADS);
        }
        mbar_init(bar_done, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_conv_x + 8 * s, CONV_PER_WARP ? 32 : CONV_THREADS);
            mbar_init(bar_conv_y + 8 * s, CONV_PER_WARP ? 32 : CONV_THREADS);
            mbar_init(bar_peer + 8 * s, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmXhi);
        tma_prefetch_desc(&tmXlo);
        tma_prefetch_desc(&tmYhi);
        tma_prefetch_desc(&tmYlo);
        if (x_ph) {
            tma_prefetch_desc(&tmX2);
            tma_prefetch_desc(&tmX3);
        }
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tc::tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
            tc::tmem_relinquish_pair();
        } else {
            tc::tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
            tc::tmem_relinquish();
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    // PAIR: both CTAs' barriers are initialised before either arrives at
    // the other's
    if constexpr (PAIR) tc::cluster_sync();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            // launched as the dependent of the split launch, the CTA set
            // itself up while it ran; the operands it writes are read only
            // after it has completed
            griddep_wait();
            int tile, k0, nk, g = 0;   // g: slabs issued so far (ring position)
            bool stop = false;
            for (int si = 0; !stop && cta_segment(SK_CTAS, KT_ALL, tiles, nsplit, rank, si, tile, k0, nk, CTAS_PER_TILE, SK_PARTS); ++si) {
                int m0, n0;
                tile_origin(tile, m0, n0);
                // PAIR: this CTA's 128 rows of A and Y_ROWS rows of B
                const int x0 = TRANS ? n0 : m0 + (int)prank * BM, y0 = TRANS ? m0 : n0 + (int)prank * Y_ROWS;
                const int zx = p.x_z ? (int)blockIdx.y : 0, zy = p.y_z ? (int)blockIdx.y : 0;
                const uint32_t tx_bytes = (x_ph ? PHASE_BYTES : (x_raw ? 1 : 2) * X_TILE) + (y_raw ? 1 : 2) * Y_TILE;
                for (int kt = 0; kt < nk; ++kt, ++g) {
                    const int s = g % STAGES;
                    if (g >= STAGES && !mbar_wait(bar_empty + 8 * s, ((g / STAGES) - 1) & 1, kStatusProducer)) {
                        *abort_flag = 1;
                        stop = true;
                        break;
                    }
                    if (*abort_flag) {
                        stop = true;
                        break;
                    }
                    const uint32_t st = stage0 + s * STAGE_BYTES;
                    const uint32_t fb = bar_full + 8 * s;
                    mbar_arrive_expect_tx(fb, tx_bytes);
                    const int kx = (k0 + kt) * BK;
                    // TMA's innermost coordinate must be 16-byte aligned (a
                    // skipped load leaves the slot's wait to run out)
                    if (!SG_IN((kx & 3) == 0 && kx < p.k)) continue;
                    if (x_ph) {
                        // the four row phases of the tile's 128 rows (32 row
                        // groups from x0 / 4), PHASE_COLS columns from kx
                        tma_load_3d(st + X_HI + 0 * PHASE_BOX, &tmXhi, kx, x0 / 4, zx, fb);
                        tma_load_3d(st + X_HI + 1 * PHASE_BOX, &tmXlo, kx, x0 / 4, zx, fb);
                        tma_load_3d(st + X_HI + 2 * PHASE_BOX, &tmX2, kx, x0 / 4, zx, fb);
                        tma_load_3d(st + X_HI + 3 * PHASE_BOX, &tmX3, kx, x0 / 4, zx, fb);
                    } else {
                        load_operand<X_MN, BM>(st + X_HI, st + X_LO, &tmXhi, &tmXlo, x_raw, x0, kx, zx, fb);
                    }
                    load_operand<Y_MN, Y_ROWS>(st + Y_HI, st + Y_LO, &tmYhi, &tmYlo, y_raw, y0, kx, zy, fb);
                }
            }
            if (*abort_flag) {
                // every copy issued must land before the CTA leaves
                for (int j = g > STAGES ? g - STAGES : 0; j < g; ++j)
                    mbar_wait(bar_full + 8 * (j % STAGES), (j / STAGES) & 1, kStatusDrain);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // PAIR: the leader issues the pair's MMAs (M = 256) and its commits
        // arrive at the barrier of the same offset in both CTAs; it waits on
        // its own barriers only
        const uint16_t pair_mask = (uint16_t)(3u << leader);
        auto commit_to = [&](uint32_t bar) {
            if constexpr (PAIR)
                tc::commit_pair(bar, pair_mask);
            else
                tc::commit(bar);
        };
        auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
            if constexpr (PAIR)
                tc::mma_tf32_pair(d, a, b, idesc, acc);
            else
                tc::mma_tf32(d, a, b, idesc, acc);
        };
        if (lane == 0 && prank == 0) {
            constexpr uint32_t idesc = tc::idesc_tf32_f32<PAIR ? 2 * BM : BM, BN, X_MN, Y_MN>();
            int tile, k0, nk, g = 0, cg = 0;   // g: slabs consumed, cg: chunks started
            bool stop = false;
            for (int si = 0; !stop && cta_segment(SK_CTAS, KT_ALL, tiles, nsplit, rank, si, tile, k0, nk, CTAS_PER_TILE, SK_PARTS); ++si) {
              for (int kt = 0; kt < nk; ++kt, ++g) {
                // each segment's slabs accumulate in chunks of CHUNK_STAGES
                // slabs, alternating between the two TMEM buffers
                const int b = cg & 1;
                const bool chunk_first = kt % CHUNK_STAGES == 0;
                const bool chunk_last = kt % CHUNK_STAGES == CHUNK_STAGES - 1 || kt == nk - 1;
                // TMEM buffer b is reused once the accumulator warps drained chunk cg - 2
                if (chunk_first && cg >= 2 &&
                    !(PAIR ? mbar_wait_cluster(bar_tempty + 8 * b, ((cg >> 1) - 1) & 1, kStatusMmaBuffer)
                           : mbar_wait(bar_tempty + 8 * b, ((cg >> 1) - 1) & 1, kStatusMmaBuffer))) {
                    *abort_flag = 1;
                    stop = true;
                    break;
                }
                const int s = g % STAGES;
                const uint32_t ph = (g / STAGES) & 1;
                if (!mbar_wait(bar_full + 8 * s, ph, kStatusMma)) {
                    *abort_flag = 1;
                    stop = true;
                    break;
                }
                // PAIR: and the peer's slab has landed and been split (its
                // signal copy's 16 bytes; they may arrive before this expect)
                if constexpr (PAIR) {
                    mbar_arrive_expect_tx(bar_peer + 8 * s, 16);
                    if (!mbar_wait(bar_peer + 8 * s, ph, kStatusMma)) {
                        *abort_flag = 1;
                        stop = true;
                        break;
                    }
                }
                // hi x hi needs only what TMA loaded; each product with a lo
                // part of a raw operand waits for the splitters to write it
                // (a phased X's hi part too)
                if (x_ph && !mbar_wait(bar_conv_x + 8 * s, ph, kStatusMma)) {
                    *abort_flag = 1;
                    stop = true;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t st = stage0 + s * STAGE_BYTES;
                const uint32_t d = tmem + (uint32_t)(b * BN);
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk)
                    mma(d, operand_desc<X_MN>(st + X_HI, kk), operand_desc<Y_MN>(st + Y_HI, kk), idesc,
                        (chunk_first && kk == 0) ? 0u : 1u);
                if (x_raw && !x_ph) {
                    if (!mbar_wait(bar_conv_x + 8 * s, ph, kStatusMma)) {
                        *abort_flag = 1;
                        stop = true;
                        break;
                    }
                    tc::fence_after_sync();
                }
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk)
                    mma(d, operand_desc<X_MN>(st + X_LO, kk), operand_desc<Y_MN>(st + Y_HI, kk), idesc, 1u);
                if (y_raw) {
                    if (!mbar_wait(bar_conv_y + 8 * s, ph, kStatusMma)) {
                        *abort_flag = 1;
                        stop = true;
                        break;
                    }
                    tc::fence_after_sync();
                }
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk)
                    mma(d, operand_desc<X_MN>(st + X_HI, kk), operand_desc<Y_MN>(st + Y_LO, kk), idesc, 1u);
                commit_to(bar_empty + 8 * s);
                if (chunk_last) {
                    commit_to(bar_tfull + 8 * b);
                    ++cg;
                }
              }
            }
            // fires once every MMA issued has completed (TMEM may then be freed)
            commit_to(bar_done);
        }
        // both CTAs of a pair: the MMAs writing this CTA's tensor memory
        // (and reading its shared memory) have completed
        if (lane == 0) mbar_wait(bar_done, 0, kStatusDrain);
        __syncwarp();
    } else if (warp >= 2 + ACC_WARPS) {
        // ------------------------------------------------------------ splitters (warps 10, 11)
        // 128-wide tiles give the tensor core ~400 cycles per slab, less
        // than one slab's split takes end to end, so there each warp splits
        // whole slabs, alternating (two in flight); 256-wide tiles leave
        // enough time for both warps to split each slab together.
        constexpr int CW = CONV_PER_WARP ? 32 : CONV_THREADS;   // threads per slab
        const int ct = CONV_PER_WARP ? lane : (int)threadIdx.x - (64 + ACC_THREADS);
        const int mine = CONV_PER_WARP ? warp - (2 + ACC_WARPS) : 0;
        int tile, k0, nk, g = 0;   // g: slab sequence position (ring position)
        // nothing to split (both operands come split), except that the odd
        // CTA of a pair still tells the leader when its slab has landed
        bool stop = !x_raw && !y_raw && !(PAIR && prank == 1);
        for (int si = 0; !stop && cta_segment(SK_CTAS, KT_ALL, tiles, nsplit, rank, si, tile, k0, nk, CTAS_PER_TILE, SK_PARTS); ++si) {
          for (int kt = 0; kt < nk; ++kt, ++g) {
            if (CONV_PER_WARP && (g % CONV_WARPS) != mine) continue;
            const int s = g % STAGES;
            const bool got = mbar_wait(bar_full + 8 * s, (g / STAGES) & 1, kStatusSplit);
            if (!got) *abort_flag = 1;
            bool quit = !got || *abort_flag != 0;
            // the odd CTA of a pair: both splitter warps meet at a named
            // barrier below on every slab, so they agree here whether to go
            // on (a wait that ran out in one warp must not leave the other
            // at that barrier)
            // so do both splitter warps of a phased X (split_phased)
            if ((PAIR && prank == 1) || (!CONV_PER_WARP && x_ph)) quit = named_barrier_or(2, CONV_THREADS, quit);
            if (quit) {
                stop = true;
                break;
            }
            // the raw slab stays as the operand's hi part (the MMA reads it
            // as hi = x with its low 13 bits dropped); lo = tf32(x - hi) goes
            // into the lo slot at the same position (the split is elementwise,
            // so the swizzled layout does not matter); X first, whose lo the
            // MMA needs first
            uint8_t *const st = smem + s * STAGE_BYTES;
            if (PAIR && prank == 0) {
                // both lo parts together (one fence), then both signals
                if (x_raw && y_raw) {
                    split_slots_lo<X_TILE, Y_TILE, CW>(st + X_HI, st + X_LO, st + Y_HI, st + Y_LO, ct);
                    tc::fence_proxy_async_smem();
                    mbar_arrive(bar_conv_x + 8 * s);
                    mbar_arrive(bar_conv_y + 8 * s);
                } else if (x_raw || y_raw) {
                    if (x_raw) split_slot_lo<X_TILE, CW>(st + X_HI, st + X_LO, ct);
                    if (y_raw) split_slot_lo<Y_TILE, CW>(st + Y_HI, st + Y_LO, ct);
                    tc::fence_proxy_async_smem();
                    mbar_arrive(x_raw ? bar_conv_x + 8 * s : bar_conv_y + 8 * s);
                }
            } else if (!PAIR) {
                // each lo part signalled to this CTA's MMA issuer as soon as
                // it is written
                if (x_raw) {
                    if (x_ph)
                        split_phased<CW>(st + X_HI, st + X_LO, (uint32_t)p.x_shift, ct);
                    else
                        split_slot_lo<X_TILE, CW>(st + X_HI, st + X_LO, ct);
                    tc::fence_proxy_async_smem();
                    mbar_arrive(bar_conv_x + 8 * s);
                }
                if (y_raw) {
                    split_slot_lo<Y_TILE, CW>(st + Y_HI, st + Y_LO, ct);
                    tc::fence_proxy_async_smem();
                    mbar_arrive(bar_conv_y + 8 * s);
                }
            } else {
                // PAIR, the odd CTA: split both halves, then one signal to the
                // leader's MMA issuer -- a 16-byte copy into the leader's
                // shared memory that completes on its barrier.  An arrival
                // from here would release at cluster scope and hold this
                // thread for ~800 cycles (measured) per slab; the copy is
                // issued and left to complete on its own.  Every writer
                // fences its lo values for the tensor core's proxy before the
                // barrier that precedes the copy.
                if (x_raw && y_raw) {
                    split_slots_lo<X_TILE, Y_TILE, CW>(st + X_HI, st + X_LO, st + Y_HI, st + Y_LO, ct);
                } else {
                    if (x_raw) split_slot_lo<X_TILE, CW>(st + X_HI, st + X_LO, ct);
                    if (y_raw) split_slot_lo<Y_TILE, CW>(st + Y_HI, st + Y_LO, ct);
                }
                tc::fence_proxy_async_smem();
                named_barrier_sync(2, CONV_THREADS);
                if (ct == 0)
                    bulk_copy_to_peer(tc::map_shared_rank(sig_pad, leader), sig_pad, 16,
                                      tc::map_shared_rank(bar_peer + 8 * s, leader));
            }
          }
        }
    } else {
        // ------------------------------------------------------------ accumulator warps (2..9)
        const int lane_grp = warp & 3;                       // TMEM lanes 32*lane_grp .. +31
        const int half = (warp - 2) >> 2;                    // columns half*128 .. +127
        const int trow = lane_grp * 32 + lane;               // this thread's row of the tile (TMEM lane)
        const uint32_t taddr = tmem + ((uint32_t)(lane_grp * 32) << 16) + (uint32_t)(half * COLS_PER_THREAD);
        float acc[COLS_PER_THREAD];
        bool ok = true;

        // Writing C.  TRANS: quad q of this thread's part of the tile at
        // (m0, n0) is rows m0 + half*COLS_PER_THREAD + 4q .. +3 of its column
        // n0 + trow of C; the 32 lanes of a warp cover 128 contiguous bytes of
        // a C row, so these go straight to C.  Stores go in blocks: the
        // block's C values (beta != 0) are loaded first, so the loads are in
        // flight together instead of each waiting behind the previous store.
        auto load_c_t = [&](int m0, int n0, int q) -> float4 {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            const int col = n0 + trow, r = m0 + half * COLS_PER_THREAD + 4 * q;
            if (col < p.n) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (r + e < p.m && SG_IN(in_matrix(Cb + (long long)(r + e) * p.ldc + col, 1, Cb, p.ldc, p.m, p.n)))
                        c[e] = Cb[(long long)(r + e) * p.ldc + col];
            }
            return make_float4(c[0], c[1], c[2], c[3]);
        };
        // C = alpha * v + beta * c for quad q (c: its C values, read when beta != 0)
        auto put_quad_t = [&](int m0, int n0, int q, float4 v, float4 c4) {
            const float alpha = p.alpha, beta = p.beta;
            const float a[4] = {v.x, v.y, v.z, v.w}, c[4] = {c4.x, c4.y, c4.z, c4.w};
            const int col = n0 + trow, r = m0 + half * COLS_PER_THREAD + 4 * q;
            if (col >= p.n) return;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (r + e < p.m && SG_IN(in_matrix(Cb + (long long)(r + e) * p.ldc + col, 1, Cb, p.ldc, p.m, p.n)))
                    Cb[(long long)(r + e) * p.ldc + col] = beta != 0.f ? fmaf(alpha, a[e], beta * c[e]) : alpha * a[e];
        };
        // Otherwise a thread's row holds 4 consecutive columns per quad, and
        // direct stores from a warp would touch 32 rows with 16 bytes each.
        // A block of 32 columns of the warp's 32 rows goes through the warp's
        // staging buffer instead and leaves as 4 rows x 128 contiguous bytes
        // per store (C, when beta != 0, is read the same way).  Chunk j of
        // row r is kept at chunk j ^ (r & 7): the row-wise writes and the
        // chunk-wise reads both touch every bank once per 128 bytes.
        auto c_at = [&](int row, int col) -> float4 {
            const float *crow = Cb + (long long)row * p.ldc;
            if (c_vec && col + 3 < p.n)
                return SG_IN(in_matrix(crow + col, 4, Cb, p.ldc, p.m, p.n)) ? *reinterpret_cast<const float4 *>(crow + col)
                                                                            : float4{};
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (col + e < p.n && SG_IN(in_matrix(crow + col + e, 1, Cb, p.ldc, p.m, p.n))) c[e] = crow[col + e];
            return make_float4(c[0], c[1], c[2], c[3]);
        };
        auto put_at = [&](int row, int col, float4 v, float4 c) {
            const float alpha = p.alpha, beta = p.beta;
            const float4 o = beta != 0.f ? make_float4(fmaf(alpha, v.x, beta * c.x), fmaf(alpha, v.y, beta * c.y),
                                                       fmaf(alpha, v.z, beta * c.z), fmaf(alpha, v.w, beta * c.w))
                                         : make_float4(alpha * v.x, alpha * v.y, alpha * v.z, alpha * v.w);
            float *crow = Cb + (long long)row * p.ldc;
            if (c_vec && col + 3 < p.n) {
                if (SG_IN(in_matrix(crow + col, 4, Cb, p.ldc, p.m, p.n))) *reinterpret_cast<float4 *>(crow + col) = o;
            } else {
                const float a[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (col + e < p.n && SG_IN(in_matrix(crow + col + e, 1, Cb, p.ldc, p.m, p.n))) crow[col + e] = a[e];
            }
        };
        // the lines of C that this thread's part of tile t covers (TRANS:
        // this warp's 32 columns of 128 rows, four rows per lane)
        auto prefetch_c = [&](int t) {
            int m0, n0;
            tile_origin(t, m0, n0);
            m0 += (int)prank * BM;
            if constexpr (TRANS) {
                const int col = n0 + lane_grp * 32;
                if (col >= p.n) return;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = m0 + half * COLS_PER_THREAD + lane + 32 * i;
                    if (row < p.m && SG_IN(in_matrix(Cb + (long long)row * p.ldc + col, 1, Cb, p.ldc, p.m, p.n)))
                        prefetch_l2(Cb + (long long)row * p.ldc + col);
                }
            } else {
                const int row = m0 + trow;
                if (row >= p.m) return;
#pragma unroll
                for (int i = 0; i < COLS_PER_THREAD / 32; ++i) {
                    const int col = n0 + half * COLS_PER_THREAD + 32 * i;
                    if (col < p.n && SG_IN(in_matrix(Cb + (long long)row * p.ldc + col, 1, Cb, p.ldc, p.m, p.n)))
                        prefetch_l2(Cb + (long long)row * p.ldc + col);
                }
            }
        };
        float4 *const stg = epi + (warp - 2) * 256;
        // v: this thread's columns half*COLS_PER_THREAD + 32*blk .. +31 of its row
        auto store_block32 = [&](int m0, int n0, int blk, const float4 (&v)[8]) {
#pragma unroll
            for (int j = 0; j < 8; ++j) stg[lane * 8 + (j ^ (lane & 7))] = v[j];
            __syncwarp();
            const int c = lane & 7;
            const int col = n0 + half * COLS_PER_THREAD + 32 * blk + 4 * c;
            const int row0 = m0 + lane_grp * 32 + (lane >> 3);   // + 4i for read i
            const bool read_c = p.beta != 0.f;
#pragma unroll
            for (int i0 = 0; i0 < 8; i0 += 4) {
                float4 cv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    cv[u] = read_c && row0 + 4 * (i0 + u) < p.m ? c_at(row0 + 4 * (i0 + u), col)
                                                                : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int rr = 4 * (i0 + u) + (lane >> 3);
                    const float4 a = stg[rr * 8 + (c ^ (rr & 7))];
                    if (row0 + 4 * (i0 + u) < p.m) put_at(row0 + 4 * (i0 + u), col, a, cv[u]);
                }
            }
            __syncwarp();   // the buffer is read before the next block overwrites it
        };
        auto store_tile = [&](int m0, int n0) {
            if constexpr (TRANS) {
                constexpr int EB = 4;   // quads per block
                const bool read_c = p.beta != 0.f;
#pragma unroll
                for (int qb = 0; qb < COLS_PER_THREAD / 4; qb += EB) {
                    float4 c[EB];
#pragma unroll
                    for (int u = 0; u < EB; ++u)
                        c[u] = read_c ? load_c_t(m0, n0, qb + u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < EB; ++u) {
                        const int q = qb + u;
                        put_quad_t(m0, n0, q, make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]),
                                   c[u]);
                    }
                }
            } else {
#pragma unroll
                for (int blk = 0; blk < COLS_PER_THREAD / 32; ++blk) {
                    float4 v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int q = 8 * blk + j;
                        v[j] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
                    }
                    store_block32(m0, n0, blk, v);
                }
            }
        };

        // stream-K: this CTA holds only part of tile t.  Publish the partial;
        // the tile's last CTA to get here adds all of the tile's partials in
        // k order (the same sum whichever CTA is last) and writes the tile.
        auto sk_partial = [&](int t, int m0, int n0) {
            // positions relative to the stream-K part of the sequence
            const int sk_tail0 = tiles / p.sk_ctas * p.sk_ctas;   // first tile shared out by slabs
            const long long T = (long long)(tiles - sk_tail0) * KT_ALL, G = p.sk_ctas;
            const long long x0 = (long long)(t - sk_tail0) * KT_ALL, x1 = x0 + KT_ALL;
            // the CTAs whose runs meet [x0, x1): g with T g / G < x1 and T (g + 1) / G > x0
            // (sk_parts >= 2: CTAs (t - sk_tail0) S + j, j = 0 .. S - 1)
            const int S = p.sk_parts;
            const int g_first = S >= 2 ? (t - sk_tail0) * S : (int)(((x0 + 1) * G - 1) / T);
            const int g_last = S >= 2 ? g_first + S - 1 : (int)((x1 * G - 1) / T);
            // a CTA's slot: 0 for the tile its run starts in, 1 for the one it
            // ends in.  Every contributor after the first starts inside the
            // tile (slot 0); only the first may have started before it.
            const int first_slot = S >= 2 || T * g_first / G >= x0 ? 0 : 1;
            const int my_slot = (int)blockIdx.x == g_first ? first_slot : 0;
            constexpr int SLOT = BM * BN / 4;   // float4s per slot
            float4 *const ws = reinterpret_cast<float4 *>(p.sk_ws);
            float4 *mine = ws + ((size_t)blockIdx.x * 2 + my_slot) * SLOT;
            const bool ws_ok = SG_IN((int)blockIdx.x < p.sk_ctas && g_first >= 0 && g_first <= g_last &&
                                     g_last < p.sk_ctas && t >= 0 && t < tiles);
#pragma unroll
            for (int q = 0; q < COLS_PER_THREAD / 4; ++q)
                if (ws_ok)
                    mine[(half * (COLS_PER_THREAD / 4) + q) * BM + trow] =
                        make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
            __threadfence();
            named_barrier_sync(1, ACC_THREADS);
            if (threadIdx.x == 64) *sk_last = ws_ok && atomicAdd(p.sk_cnt + t, 1) == g_last - g_first;
            named_barrier_sync(1, ACC_THREADS);
            const bool last = *sk_last != 0;
            named_barrier_sync(1, ACC_THREADS);   // the flag is read before it is next written
            if (!last) return;
            __threadfence();
            // the other contributors' partials were written long before
            // (their runs reach this tile first) and have mostly left L2:
            // bring them back in bulk while the first block's loads start
            if (threadIdx.x == 64) {
                for (int g = g_first; g < g_last; ++g) {
                    const float4 *src = g == g_first ? ws + ((size_t)g_first * 2 + first_slot) * SLOT
                                                     : ws + (size_t)g * 2 * SLOT;
                    bulk_prefetch_l2(src, SLOT * 16u);
                }
            }
            // blocks of QB quads: each contributor's QB loads are in flight
            // together (one L2 round trip per block and contributor)
            constexpr int QB = 8;   // = one 32-column block of store_block32
            const float4 *first = ws + ((size_t)g_first * 2 + first_slot) * SLOT;
#pragma unroll 1
            for (int qb = 0; qb < COLS_PER_THREAD / 4; qb += QB) {
                const int idx0 = (half * (COLS_PER_THREAD / 4) + qb) * BM + trow;
                float4 sum[QB];
#pragma unroll
                for (int u = 0; u < QB; ++u) sum[u] = __ldcg(first + idx0 + u * BM);
#pragma unroll 1
                for (int g = g_first + 1; g <= g_last; ++g) {
                    const float4 *src = ws + (size_t)g * 2 * SLOT + idx0;
                    float4 v[QB];
#pragma unroll
                    for (int u = 0; u < QB; ++u) v[u] = __ldcg(src + u * BM);
#pragma unroll
                    for (int u = 0; u < QB; ++u) {
                        sum[u].x += v[u].x;
                        sum[u].y += v[u].y;
                        sum[u].z += v[u].z;
                        sum[u].w += v[u].w;
                    }
                }
                if constexpr (TRANS) {
                    const bool read_c = p.beta != 0.f;
                    float4 c[QB];
#pragma unroll
                    for (int u = 0; u < QB; ++u)
                        c[u] = read_c ? load_c_t(m0, n0, qb + u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < QB; ++u) put_quad_t(m0, n0, qb + u, sum[u], c[u]);
                } else {
                    store_block32(m0, n0, qb / QB, sum);
                }
            }
        };

        int tile, k0, nk, cg = 0;   // cg: chunks drained so far
        for (int si = 0; cta_segment(SK_CTAS, KT_ALL, tiles, nsplit, rank, si, tile, k0, nk, CTAS_PER_TILE, SK_PARTS); ++si) {
#pragma unroll
            for (int j = 0; j < COLS_PER_THREAD; ++j) acc[j] = 0.f;
            const int nc = (nk + CHUNK_STAGES - 1) / CHUNK_STAGES;
            for (int c = 0; c < nc && ok; ++c, ++cg) {
                // beta != 0: while the tile's last chunk accumulates, bring
                // the lines of C this warp will read (the old values) into
                // L2, so the epilogue's loads of them do not go to DRAM
                if (c == nc - 1 && p.beta != 0.f) prefetch_c(tile);
                const int b = cg & 1;
                const bool got = mbar_wait(bar_tfull + 8 * b, (cg >> 1) & 1, kStatusAccumulate);
                if (!got) *abort_flag = 1;
                // PAIR: the accumulator threads meet at a named barrier below
                // on every chunk, so they agree here whether to go on
                const bool quit = PAIR ? named_barrier_or(3, ACC_THREADS, !got) : !got;
                if (quit) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
#pragma unroll
                for (int q = 0; q < COLS_PER_THREAD / 16; ++q) {
                    uint32_t v[16];
                    tc::ld_32x32b_x16(taddr + (uint32_t)(b * BN + q * 16), v);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[q * 16 + i] += __uint_as_float(v[i]);
                }
                tc::fence_before_sync();
                if constexpr (PAIR) {
                    // one arrival per CTA at the leader's barrier, after every
                    // accumulator thread's loads of the buffer have completed
                    named_barrier_sync(4, ACC_THREADS);
                    if (threadIdx.x == 64) arrive_leader(bar_tempty + 8 * b);
                } else {
                    mbar_arrive(bar_tempty + 8 * b);
                }
            }
            // leave together (the stream-K hand-off below synchronises
            // these 256 threads, and a wait that ran out may have stopped
            // only some of them)
            if (named_barrier_or(1, ACC_THREADS, !ok || *abort_flag != 0)) break;
            int m0, n0;
            tile_origin(tile, m0, n0);
            m0 += (int)prank * BM;   // PAIR: this CTA's 128 rows of the 256-row tile
            if (nsplit > 1) {
                // park the partial tile in this CTA's (now idle) stage memory,
                // rows PART_PITCH floats apart (4 banks apart: conflict-free)
                float *part = reinterpret_cast<float *>(smem) + trow * PART_PITCH + half * COLS_PER_THREAD;
                const bool part_ok = SG_IN(trow * PART_PITCH + half * COLS_PER_THREAD + COLS_PER_THREAD <= BM * PART_PITCH);
#pragma unroll
                for (int q = 0; q < COLS_PER_THREAD / 4; ++q)
                    if (part_ok)
                        reinterpret_cast<float4 *>(part)[q] =
                            make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
            } else if (sk && nk < KT_ALL) {
                sk_partial(tile, m0, n0);
            } else {
                store_tile(m0, n0);
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (nsplit > 1) {
        // ------------------------------------------------------------ cluster reduction
        // every partial is parked; CTA `rank` sums rows [r0, r1) of the tile
        // over the cluster's CTAs in rank order (a fixed order: the result
        // does not depend on timing) and writes them to C.  A thread's
        // values (at most MAXIT float4 of the tile) are gathered rank by
        // rank with all of a rank's remote loads in flight together (the
        // abort flags with the first rank's), then C's values (beta != 0),
        // also all at once: a few load latencies in all, not two per float4.
        // Once its remote values are in registers a thread tells the cluster
        // (the second barrier's arrival, which need not wait for the stores);
        // it waits for the others only before leaving, so no CTA leaves
        // while another may still read its partial.
        tc::cluster_sync();
        const uint32_t part0 = smem_u32(smem);
        const uint32_t abort_addr = smem_u32(const_cast<int *>(abort_flag));
        const int r0 = (int)(BM * rank / nsplit), r1 = (int)(BM * (rank + 1) / nsplit);
        const int nrows = r1 - r0, total = nrows * (BN / 4);
        constexpr int MAXIT = ((BM / 2) * (BN / 4) + NTHREADS - 1) / NTHREADS;   // nsplit >= 2
        const float alpha = p.alpha, beta = p.beta;
        // float4 `it` of this thread: tile row r, columns 4 c4 .. +3 (TRANS:
        // consecutive threads take consecutive tile rows (= columns of C),
        // so the stores below stay coalesced)
        uint32_t off[MAXIT];
#pragma unroll
        for (int it = 0; it < MAXIT; ++it) {
            const int idx = (int)threadIdx.x + it * NTHREADS;
            const int r = TRANS ? r0 + idx % nrows : r0 + idx / (BN / 4);
            const int c4 = TRANS ? idx / nrows : idx % (BN / 4);
            off[it] = part0 + (uint32_t)(r * PART_PITCH + 4 * c4) * 4u;
            // (an index past this thread's share is never used)
            if (idx < total && !SG_IN(r >= 0 && r < BM && 4 * c4 + 4 <= BN)) off[it] = part0;
        }
        int flags[8];
#pragma unroll
        for (uint32_t q = 0; q < 8; ++q) flags[q] = q < nsplit ? tc::ld_cluster_s32(tc::map_shared_rank(abort_addr, q)) : 0;
        float4 sum[MAXIT], v[MAXIT];
#pragma unroll
        for (int it = 0; it < MAXIT; ++it)
            if ((int)threadIdx.x + it * NTHREADS < total) sum[it] = tc::ld_cluster_v4(tc::map_shared_rank(off[it], 0));
        for (uint32_t q = 1; q < nsplit; ++q) {
#pragma unroll
            for (int it = 0; it < MAXIT; ++it)
                if ((int)threadIdx.x + it * NTHREADS < total) v[it] = tc::ld_cluster_v4(tc::map_shared_rank(off[it], q));
#pragma unroll
            for (int it = 0; it < MAXIT; ++it) {
                if ((int)threadIdx.x + it * NTHREADS < total) {
                    sum[it].x += v[it].x;
                    sum[it].y += v[it].y;
                    sum[it].z += v[it].z;
                    sum[it].w += v[it].w;
                }
            }
        }
        int any_abort = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) any_abort |= flags[q];
        __syncwarp();
        tc::cluster_arrive_relaxed();
        if (!any_abort) {
            // C's old values (beta != 0) into v: TRANS, four rows of one
            // column of C; otherwise four columns of one row
#pragma unroll
            for (int it = 0; it < MAXIT; ++it) {
                const int idx = (int)threadIdx.x + it * NTHREADS;
                v[it] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (beta == 0.f || idx >= total) continue;
                const int r = TRANS ? r0 + idx % nrows : r0 + idx / (BN / 4);
                const int c4 = TRANS ? idx / nrows : idx % (BN / 4);
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                if constexpr (TRANS) {
                    const int cc = cl_n0 + r, rr = cl_m0 + 4 * c4;   // column of C, first of 4 rows
                    if (cc < p.n) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (rr + e < p.m && SG_IN(in_matrix(Cb + (long long)(rr + e) * p.ldc + cc, 1, Cb, p.ldc, p.m, p.n)))
                                c[e] = Cb[(long long)(rr + e) * p.ldc + cc];
                    }
                } else {
                    const int row = cl_m0 + r, col = cl_n0 + 4 * c4;
                    if (row < p.m) {
                        const float *crow = Cb + (long long)row * p.ldc;
                        if (c_vec && col + 3 < p.n && SG_IN(in_matrix(crow + col, 4, Cb, p.ldc, p.m, p.n))) {
                            const float4 c4v = *reinterpret_cast<const float4 *>(crow + col);
                            c[0] = c4v.x;
                            c[1] = c4v.y;
                            c[2] = c4v.z;
                            c[3] = c4v.w;
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (col + e < p.n && SG_IN(in_matrix(crow + col + e, 1, Cb, p.ldc, p.m, p.n)))
                                    c[e] = crow[col + e];
                        }
                    }
                }
                v[it] = make_float4(c[0], c[1], c[2], c[3]);
            }
#pragma unroll
            for (int it = 0; it < MAXIT; ++it) {
                const int idx = (int)threadIdx.x + it * NTHREADS;
                if (idx >= total) continue;
                const int r = TRANS ? r0 + idx % nrows : r0 + idx / (BN / 4);
                const int c4 = TRANS ? idx / nrows : idx % (BN / 4);
                const float a[4] = {sum[it].x, sum[it].y, sum[it].z, sum[it].w};
                const float c[4] = {v[it].x, v[it].y, v[it].z, v[it].w};
                float o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = beta != 0.f ? fmaf(alpha, a[e], beta * c[e]) : alpha * a[e];
                if constexpr (TRANS) {
                    const int cc = cl_n0 + r, rr = cl_m0 + 4 * c4;
                    if (cc >= p.n) continue;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (rr + e < p.m && SG_IN(in_matrix(Cb + (long long)(rr + e) * p.ldc + cc, 1, Cb, p.ldc, p.m, p.n)))
                            Cb[(long long)(rr + e) * p.ldc + cc] = o[e];
                    continue;
                }
                const int row = cl_m0 + r, col = cl_n0 + 4 * c4;
                if (row >= p.m) continue;
                float *crow = Cb + (long long)row * p.ldc;
                if (c_vec && col + 3 < p.n) {
                    if (SG_IN(in_matrix(crow + col, 4, Cb, p.ldc, p.m, p.n)))
                        *reinterpret_cast<float4 *>(crow + col) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (col + e < p.n && SG_IN(in_matrix(crow + col + e, 1, Cb, p.ldc, p.m, p.n))) crow[col + e] = o[e];
                }
            }
        }
        __syncwarp();
        tc::cluster_wait();
    }
    // PAIR: neither CTA leaves (or frees its tensor memory) while the other
    // may still arrive at its barriers
    if constexpr (PAIR) tc::cluster_sync();
    if (warp == 1) {
        tc::fence_after_sync();
        if constexpr (PAIR)
            tc::tmem_dealloc_pair(tmem, TMEM_COLS);
        else
            tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace tf32x3
}  // namespace sgemm_gb300
