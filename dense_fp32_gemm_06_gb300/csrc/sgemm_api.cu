// C ABI of the GB300 SGEMM library: argument checks, launch planning and
// kernel launches.  Declared in include/sgemm_gb300.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/sgemm_gb300.h"
#include "reduce_sum.cuh"
#include "units.h"

using namespace sgemm_gb300;

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    // clusters of S CTAs (S = 2..8) of the tensor-core kernel that fit on the
    // device at once, for the 256- and 128-wide tiles ([0] and [1]); [2][2]:
    // CTA pairs of the Pair configuration
    int max_clusters[3][9] = {};
    // stream-ordered pool of the tensor-core path's scratch; keeps up to
    // its release threshold mapped between calls (the default pool's
    // threshold is 0: every synchronize would unmap the scratch and the next
    // call map it again, ~0.1 ms each time)
    cudaMemPool_t pool = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

// Kernel ids in sgemm_plan::kernel.
constexpr int kKernelFfmaCpAsync = 0;
constexpr int kKernelScale = 1;
constexpr int kKernelTf32x3 = 2;
// GB300's L2 (the plans are for sm_103a devices; host-only plans too)
constexpr double kL2Bytes = 129e6;

int fail_cuda(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return SGEMM_STATUS_CUDA_ERROR;
}

// One-time per-device set-up: SM count and kernel attributes.
int device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return fail_cuda(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail_cuda(e);
        if ((e = units::ffma_attrs()) != cudaSuccess) return fail_cuda(e);
        if ((e = units::tc_wide_attrs()) != cudaSuccess) return fail_cuda(e);
        if ((e = units::tc_narrow_attrs()) != cudaSuccess) return fail_cuda(e);
        if ((e = units::tc_trans_attrs()) != cudaSuccess) return fail_cuda(e);
        if ((e = units::tc_pair_attrs()) != cudaSuccess) return fail_cuda(e);
        for (int S = 2; S <= 8; ++S) {
            if ((e = units::tc_wide_clusters(S, &d.max_clusters[0][S])) != cudaSuccess) return fail_cuda(e);
            if ((e = units::tc_narrow_clusters(S, &d.max_clusters[1][S])) != cudaSuccess) return fail_cuda(e);
        }
        if ((e = units::tc_pair_clusters(2, &d.max_clusters[2][2])) != cudaSuccess) return fail_cuda(e);
        if (d.pool == nullptr) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            if ((e = cudaMemPoolCreate(&d.pool, &props)) != cudaSuccess) {
                d.pool = nullptr;
                return fail_cuda(e);
            }
            unsigned long long keep_mb = 2048;
            if (const char *env = std::getenv("SGEMM_GB300_POOL_KEEP_MB"))
                if (env[0] >= '0' && env[0] <= '9') keep_mb = std::strtoull(env, nullptr, 10);
            cuuint64_t thr = (cuuint64_t)keep_mb << 20;
            if ((e = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &thr)) != cudaSuccess)
                return fail_cuda(e);
        }
        if (g_encode_tiled == nullptr) {
            cudaDriverEntryPointQueryResult q;
            void *fn = nullptr;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
                return fail_cuda(e != cudaSuccess ? e : cudaErrorSymbolNotFound);
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    *out = &d;
    return SGEMM_STATUS_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int imax(int a, int b) { return a > b ? a : b; }

// A strided batch of problems: problem b uses A + b*sa, B + b*sb, C + b*sc.
struct Batch {
    int count = 1;
    long long sa = 0, sb = 0, sc = 0;
};

// BLAS-style argument check; returns the 1-based position of the first bad
// argument, or 0.
// op_a / op_b: SGEMM_OP_N (A stored m x k, B stored k x n) or SGEMM_OP_T
// (A stored k x m, B stored n x k); positions are those of sgemm().
int check_args(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb,
               const float *C, int ldc, int op_a = SGEMM_OP_N, int op_b = SGEMM_OP_N) {
    if (m < 0) return 1;
    if (n < 0) return 2;
    if (k < 0) return 3;
    const bool need_ab = (long long)m * n * k > 0 && alpha != 0.f;
    if (need_ab && (A == nullptr || !aligned(A, 4))) return 5;
    if (lda < imax(1, op_a == SGEMM_OP_N ? k : m)) return 6;
    if (need_ab && (B == nullptr || !aligned(B, 4))) return 7;
    if (ldb < imax(1, op_b == SGEMM_OP_N ? n : k)) return 8;
    if ((long long)m * n > 0 && (C == nullptr || !aligned(C, 4))) return 10;
    if (ldc < imax(1, n)) return 11;
    return 0;
}

// max_clusters: the device's cluster capacity table (DeviceState), or NULL
// for a host-only plan, which assumes 8 GPCs of num_sms / 8 SMs.
// Whether the tensor-core GEMM can read an operand as stored, by TMA: a
// 16-byte aligned base and 16-byte rows, and in a batch either one matrix
// for all problems (stride 0) or problems that do not overlap, 16 bytes apart.
// `outer` x `ld` is the stored matrix (rows x row pitch).
bool tma_readable(const void *X, long long ld, long long outer, int batch, long long stride) {
    if (!aligned(X, 16) || ld % 4 != 0) return false;
    if (batch > 1 && stride != 0 && (stride % 4 != 0 || stride < outer * ld)) return false;
    return true;
}

// Whether a K-major operand TMA cannot read as stored can be read in row
// phases (rows j, j + 4, ...: 4 * ld floats apart, a multiple of 16 bytes):
// always for one matrix; in a batch, one matrix for all problems or
// problems that do not overlap, a multiple of 4 floats apart (each phase
// then has the same shift in every problem).
bool phase_readable(long long outer, long long ld, int batch, long long stride) {
    return !(batch > 1 && stride != 0 && (stride % 4 != 0 || stride < outer * ld));
}

// The tensor-core plan on CTA pairs: 256 x 256 tiles of two CTAs each, whole
// tiles (no split-K, no stream-K); the operand sources stay as planned.
void set_pair_plan(int m, int n, int k, sgemm_plan *pl) {
    pl->pair = 1;
    pl->trans = 0;
    pl->persistent = 0;
    pl->bm = pl->bn = tf32x3::Pair::BN;
    pl->split_k = 1;
    pl->stream_k = 0;
    pl->sk_parts = 0;
    pl->stages = tf32x3::Pair::STAGES;
    pl->smem_bytes = tf32x3::Pair::SMEM_BYTES;
    const int tm = (m + pl->bm - 1) / pl->bm, tn = (n + pl->bn - 1) / pl->bn;
    pl->tiles = tm * tn;
    pl->grid = 2 * pl->tiles;
    pl->k_tiles = (k + tf32x3::BK - 1) / tf32x3::BK;
    pl->group_m = tm < 8 ? tm : 8;
}

int plan(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
         const float *C, int ldc, int path, int num_sms, sgemm_plan *pl, const int (*max_clusters)[9] = nullptr,
         int op_a = SGEMM_OP_N, int op_b = SGEMM_OP_N, int batch = 1, bool allow_sk = true,
         long long stride_a = 0, long long stride_b = 0) {
    (void)beta;
    std::memset(pl, 0, sizeof(*pl));
    if (path != SGEMM_PATH_AUTO && path != SGEMM_PATH_FFMA && path != SGEMM_PATH_TF32X3)
        return SGEMM_STATUS_BAD_PATH;
    if (int bad = check_args(m, n, k, alpha, A, lda, B, ldb, C, ldc, op_a, op_b)) return bad;
    if (m == 0 || n == 0) return SGEMM_STATUS_OK;
    if (num_sms <= 0) num_sms = 1;
    pl->op_a = op_a;
    pl->op_b = op_b;
    // AUTO: the tensor-core path from 2^20 multiply-adds with k >= 64 (it is
    // ~5x the FFMA rate at 2048^3 and beyond, and its two launches already
    // beat the FFMA kernel's 128 x 128 tiles at 128^3: 16 against 19 us,
    // whole call, L2 flushed) and for long k (its chunked accumulation holds
    // the bound where a plain sequential FP32 sum over k drifts); the FFMA
    // path for tiny problems (64^3: 13 against 14 us) and for k < 64, where
    // the split passes cost more than they save (4096 x 4096 x 32: 35.5
    // against 40.6 us).
    const long long mnk = (long long)m * n * k;
    const bool use_tc = path == SGEMM_PATH_TF32X3 ||
                        (path == SGEMM_PATH_AUTO && ((mnk >= (1LL << 20) && k >= 64) || k > 8192));
    pl->path = use_tc ? SGEMM_PATH_TF32X3 : SGEMM_PATH_FFMA;
    pl->split_k = 1;
    pl->c_vec = aligned(C, 16) && (ldc % 4) == 0;
    if (k == 0 || alpha == 0.f) {
        pl->kernel = kKernelScale;
        pl->threads = 256;
        const long long total = (long long)m * n;
        long long blocks = (total + 255) / 256;
        pl->grid = (int)(blocks < 4096 ? blocks : 4096);
        pl->c_vec = 0;
        return SGEMM_STATUS_OK;
    }
    if (use_tc) {
        pl->kernel = kKernelTf32x3;
        pl->bm = tf32x3::BM;
        pl->bk = tf32x3::BK;
        pl->threads = tf32x3::THREADS;
        pl->b_vec = 1;
        // Tile shape and split-K factor S: the pair with the smallest
        // estimated time waves x ceil(KT / S) x (slab time) (+ the cost of a
        // split's cluster reduction).  Slab times, measured on GB300: a
        // 256-wide slab ~0.5 us, a 128-wide one ~0.375 us (1.5x the time per
        // FLOP), a transposed 256 x 128 one ~0.66 us (split-K cases: its
        // 16 KB of A to split and its column-wise stores); a split adds
        // ~2 us + 0.5 us per CTA of the cluster (fitted to whole calls and
        // split-K sweeps: 256 x 256 x 8192 over S = 1..8, 384^3, 500 x 500
        // x 300).  Units below: 1/32 us.
        // Waves count CTAs against the SMs (S = 1) or
        // clusters against the clusters that fit at once (S > 1); a split
        // must fit in one wave and leave each CTA >= 4 slabs (64 k).
        const int tiles_m = (m + pl->bm - 1) / pl->bm;
        const long long KT = (k + tf32x3::BK - 1) / tf32x3::BK;
        // tuning overrides for benchmarks and tests: SGEMM_GB300_TILE_N (128
        // or 256) and SGEMM_GB300_SPLIT_K (1..8) pin the choice below
        const char *env_bn = std::getenv("SGEMM_GB300_TILE_N");
        const char *env_s = std::getenv("SGEMM_GB300_SPLIT_K");
        const int force_bn = env_bn ? std::atoi(env_bn) : 0;
        const int force_s = env_s ? std::atoi(env_s) : 0;
        // Candidates: 256-wide tiles, 128-wide tiles, and for n <= 128 the
        // transposed tile (C^T = B^T A^T: 256 rows of C by 128 columns), which
        // keeps the MMA 256 wide -- a 128 x 128 x 8 MMA takes about as long
        // as a 128 x 256 x 8 one.  SGEMM_GB300_TRANS (0 / 1) pins the last.
        const char *env_tr = std::getenv("SGEMM_GB300_TRANS");
        const int force_tr = env_tr && (env_tr[0] == '0' || env_tr[0] == '1') ? env_tr[0] - '0' : -1;
        // Stream-K: one persistent CTA per SM; the full waves of tiles run
        // as whole tiles, the tiles of the last, partial wave are shared out
        // evenly by slabs (so no SM idles in it); a tile split between CTAs
        // is finished by the last of them through a workspace (~10 us).  Only
        // for one problem and when the last wave has enough tiles that a
        // tile meets few CTAs.  SGEMM_GB300_STREAM_K (0 / 1) pins it.
        const char *env_sk = std::getenv("SGEMM_GB300_STREAM_K");
        const int force_sk = env_sk && (env_sk[0] == '0' || env_sk[0] == '1') ? env_sk[0] - '0' : -1;
        long long best = -1;
        int best_bn = tf32x3::Wide::BN, best_s = 1;
        bool best_tr = false, best_sk = false;
        auto consider = [&](long long cost, int bn, int S, bool tr, bool skc) {
            // a pinned stream-K choice beats every other candidate
            const bool better = force_sk == 1 && skc != best_sk ? skc : (best < 0 || cost < best);
            if (better) {
                best = cost;
                best_bn = bn;
                best_s = S;
                best_tr = tr;
                best_sk = skc;
            }
        };
        for (int cand = 0; cand < 3; ++cand) {
            const bool tr = cand == 2;
            const int bn = cand == 1 ? tf32x3::Narrow::BN : tf32x3::Wide::BN;
            if (tr) {
                if (force_tr == 0 || n > tf32x3::BM || (force_bn != 0 && force_tr != 1)) continue;
            } else if (force_tr == 1 && n <= tf32x3::BM) {
                continue;
            } else if (force_bn == tf32x3::Wide::BN || force_bn == tf32x3::Narrow::BN) {
                if (bn != force_bn) continue;
            } else if (bn == tf32x3::Wide::BN && n <= tf32x3::Narrow::BN) {
                continue;
            }
            const int wi = bn == tf32x3::Wide::BN ? 0 : 1;
            const long long slab = tr ? 21 : bn == tf32x3::Wide::BN ? 16 : 12;
            const long long tiles = tr ? (long long)((m + tf32x3::Wide::BN - 1) / tf32x3::Wide::BN) *
                                             ((n + tf32x3::BM - 1) / tf32x3::BM) * (batch > 0 ? batch : 1)
                                       : (long long)tiles_m * ((n + bn - 1) / bn) * (batch > 0 ? batch : 1);
            for (int S = 1; S <= 8; ++S) {
                if (force_s >= 1 && force_s <= 8) {
                    if (S != force_s) continue;
                } else if (S > 1 && KT / S < 4) {
                    break;
                }
                long long slots = num_sms;   // CTAs (S = 1) or clusters (S > 1) resident at once
                if (S > 1) {
                    slots = max_clusters ? max_clusters[wi][S] : 8LL * ((num_sms / 8) / S);
                    // a split only pays when all of its clusters run in one wave
                    if (slots <= 0 || (tiles > slots && !(force_s >= 1 && force_s <= 8))) continue;
                }
                const long long waves = (tiles + slots - 1) / slots;
                const long long cost = waves * ((KT + S - 1) / S) * slab + (S > 1 ? 64 + 16 * S : 0);
                consider(cost, bn, S, tr, false);
            }
            // stream-K: W = tiles / G full waves of whole tiles, then the R
            // remaining tiles' slabs shared out evenly (every CTA must get at
            // least one slab of them: R x KT >= G, and a shared tile meets a
            // few CTAs only: 4 R >= G).  Measured: the fix-up of a shared tile
            // costs ~10 us, twice when a CTA's share is shorter than a tile
            // (it then holds parts of two).  Against persistent whole tiles
            // (interleaved, whole calls): 4096^3 17 % faster, 8192 x 8192 x
            // 4096 1.88 against 1.94 ms, 6144^3 1.71 against 1.76, 12288 x
            // 8192 x 4096 2.87 against 2.96, 8192^3 3.80 against 3.82.
            const long long W = tiles / num_sms, R = tiles - W * num_sms;
            if (allow_sk && force_sk != 0 && batch == 1 && !(force_s >= 1 && force_s <= 8) && R > 0 &&
                R * KT >= num_sms && (4 * R >= num_sms || force_sk == 1)) {
                const long long share = (R * KT + num_sms - 1) / num_sms;
                consider(W * KT * slab + share * slab + (share < KT ? 640 : 320), bn, 1, tr, true);
            }
        }
        // Each operand is read by the GEMM as the caller stored it whenever
        // TMA can read it (tma_readable): the GEMM's two splitter warps turn
        // each raw slab into its TF32 lo part in shared memory and the MMA
        // reads the raw slab as the hi part, so the call needs no split pass
        // and no scratch memory for that operand.  Otherwise the split pass
        // writes the operand's hi and lo parts into scratch first.
        // SGEMM_GB300_SPLIT_A_IN / SGEMM_GB300_SPLIT_B_IN = 0 force the split
        // pass (tests and measurements).
        // B's split, though, is ~1.6x the work of A's per slab (the tile's
        // 256 n-rows against 128 m-rows), and on 128 x 256 tiles the
        // splitter warps' shared-memory traffic then holds up the tensor
        // core (measured, whole call, L2 flushed: 8192^3 5.8 against 3.7 ms
        // with B split by the split pass; 2048^3 118 against 82 us), while
        // for small problems the split pass's launch and round trip cost
        // more (256^3 14.7 against 16.3 us; 1000 x 1500 x 780 35.8 against
        // 36.6).  So B is read as stored for m*n*k <= 2^31 only.
        const char *env_ain = std::getenv("SGEMM_GB300_SPLIT_A_IN");
        const char *env_bin = std::getenv("SGEMM_GB300_SPLIT_B_IN");
        const bool a_tma = tma_readable(A, lda, op_a == SGEMM_OP_N ? m : k, batch, stride_a);
        const bool b_tma = tma_readable(B, ldb, op_b == SGEMM_OP_N ? k : n, batch, stride_b);
        const bool b_small = (long long)m * n * k * (batch > 0 ? batch : 1) <= (1LL << 31);
        // an A that TMA cannot read as one tensor (rows not 16 bytes apart,
        // a misaligned base) on untransposed tiles is read in four row
        // phases, each of which TMA can read, and put in place and split by
        // the GEMM's splitter warps
        const bool a_phased = !a_tma && op_a == SGEMM_OP_N && !best_tr && phase_readable(m, lda, batch, stride_a);
        pl->a_in_kernel = (a_tma || a_phased) && !(env_ain && env_ain[0] == '0');
        pl->b_in_kernel = b_tma && (env_bin && (env_bin[0] == '0' || env_bin[0] == '1') ? env_bin[0] == '1' : b_small);
        pl->threads = tf32x3::THREADS;
        // CTA pairs (cta_group::2): 256 x 256 tiles, each CTA staging (and,
        // for operands read as stored, splitting) 128 rows of A and 128 of
        // B; whole tiles only (no split-K, no stream-K).
        // SGEMM_GB300_PAIR = 1 asks for it where it applies.
        // The default takes pairs where they are the faster plan and spare
        // B's split pass: above 2^31 multiply-adds (where B would be split
        // first), both operands read as stored, and 256 x 256 tiles that fill
        // at least three quarters of the device's pair slots in one wave
        // (measured, whole call, L2 flushed: 2048^3 81.9 against 83.9 us; at
        // 8192^3, many waves, 4.02 against 3.71 ms, and at 4096^3 against
        // stream-K 622 against 527 us, so those keep single CTAs).
        // SGEMM_GB300_PAIR = 1 / 0 pins the choice (1: wherever the tiles are
        // not transposed).
        const char *env_pair = std::getenv("SGEMM_GB300_PAIR");
        const long long pair_tiles = (long long)((m + 255) / 256) * ((n + 255) / 256) * (batch > 0 ? batch : 1);
        const long long pair_slots = max_clusters ? max_clusters[2][2] : num_sms / 2;
        // (any pin of the single-CTA plan -- tile width, split-K, transposed
        // tiles, stream-K -- keeps that plan)
        const bool pinned = force_bn != 0 || (force_s >= 1 && force_s <= 8) || force_tr != -1 || force_sk != -1;
        const bool pair_auto = a_tma && b_tma && !b_small && pl->a_in_kernel && !(env_bin && env_bin[0] == '0') &&
                               !pinned && pair_tiles <= pair_slots && 4 * pair_tiles >= 3 * pair_slots;
        if (!best_tr && (env_pair ? env_pair[0] == '1' : pair_auto)) {
            if (!env_pair) pl->b_in_kernel = 1;
            if (!a_tma) pl->a_in_kernel = 0;   // pairs read A by TMA or take it split
            set_pair_plan(m, n, k, pl);
            return SGEMM_STATUS_OK;
        }
        const bool narrow = best_bn == tf32x3::Narrow::BN;
        pl->trans = best_tr;
        // bm x bn: the tile of C (256 x 128 when transposed)
        pl->bm = best_tr ? tf32x3::Wide::BN : tf32x3::BM;
        pl->bn = best_tr ? tf32x3::BM : best_bn;
        pl->split_k = best_s;
        pl->stream_k = best_sk ? num_sms : 0;
        pl->stages = narrow ? tf32x3::Narrow::STAGES : tf32x3::Wide::STAGES;
        pl->smem_bytes = narrow ? tf32x3::Narrow::SMEM_BYTES : tf32x3::Wide::SMEM_BYTES;
        const int tiles_mt = (m + pl->bm - 1) / pl->bm;
        const int tiles_n = (n + pl->bn - 1) / pl->bn;
        pl->tiles = tiles_mt * tiles_n;
        pl->grid = best_sk ? num_sms : pl->tiles * pl->split_k;
        // whole tiles of more than one wave: one persistent CTA per SM takes
        // tiles g, g + sms, ... in turn, a tile's epilogue overlapping the
        // next one's first chunks (measured, whole call, L2 flushed:
        // 8192^3 3.83 against 3.89 ms, 8192 x 8192 x 4096 1.91 against
        // 1.99, 16384 x 4096 x 4096 1.89 against 1.96).
        // SGEMM_GB300_PERSIST (0 / 1) pins it.
        const char *env_ps = std::getenv("SGEMM_GB300_PERSIST");
        const int force_ps = env_ps && (env_ps[0] == '0' || env_ps[0] == '1') ? env_ps[0] - '0' : -1;
        if (!best_sk && best_s == 1 && batch == 1 && pl->tiles > num_sms && force_ps != 0) {
            pl->persistent = 1;
            pl->grid = num_sms;
        }
        // stream-K after at least two full waves, with S = sms / R >= 2 for
        // the R remaining tiles: each of those is cut into S equal k parts
        // (CTA i S + j takes part j of remaining tile i) rather than the
        // slab sequence into equal runs, so that CTAs on one tile row
        // (column) read the same k range of its A (B) panel at once and
        // share it in L2 -- equal runs start at unrelated k offsets, and that
        // tail then streams every panel from DRAM.
        // SGEMM_GB300_SK_PARTS (0 / 1) pins it.
        if (best_sk) {
            const char *env_sp = std::getenv("SGEMM_GB300_SK_PARTS");
            const long long W = pl->tiles / num_sms, R = pl->tiles - W * num_sms;
            const int S = R > 0 ? (int)(num_sms / R) : 0;
            const bool parts = env_sp && (env_sp[0] == '0' || env_sp[0] == '1') ? env_sp[0] == '1' : W >= 2;
            if (parts && S >= 2 && KT >= S) pl->sk_parts = S;
        }
        pl->k_tiles = (int)KT;
        // Raster groups: a wave of G = sms CTAs covers g tile rows x G / g
        // tile columns, and reads g A panels (BM rows of k) and G / g B
        // panels (BN rows) -- 4 bytes a value as stored, 8 split -- which
        // costs least near g = sqrt(G x B panel / A panel): ~25 for 128 x 256
        // tiles with B split first.  Where the operands as read exceed twice
        // L2 (DRAM-streamed), 24 tile rows; otherwise 8, which keeps the
        // panels of the CTAs running at once together in L2.  Measured
        // (whole calls, interleaved, L2 flushed): 8192 x 8192 x 4096 1880
        // against 1920 us, 16384 x 8192 x 4096 3744 against 3818; 8192^3
        // DRAM per launch 5.27 -> ~3.4 GB and the 300-step bench line, held
        // at the power cap, 294.2 - 294.5 against 287.5 - 289.6 TFLOPS
        // (higher clocks at the same power); 4096^3 (operands ~1.5x L2) 0.9 %
        // slower with 24.  SGEMM_GB300_GROUP_M (1 .. 64) pins it.
        const double op_bytes = (double)m * k * (pl->a_in_kernel ? 4 : 8) * (batch > 0 ? batch : 1) +
                                (double)n * k * (pl->b_in_kernel ? 4 : 8) * (batch > 0 ? batch : 1);
        const char *env_gm = std::getenv("SGEMM_GB300_GROUP_M");
        const int gm = env_gm && std::atoi(env_gm) >= 1 && std::atoi(env_gm) <= 64 ? std::atoi(env_gm)
                       : op_bytes > 2.0 * kL2Bytes                                    ? 24
                                                                                      : 8;
        pl->group_m = tiles_mt < gm ? tiles_mt : gm;
        return SGEMM_STATUS_OK;
    }
    pl->kernel = kKernelFfmaCpAsync;
    // 8 x 16 outputs per thread (128 threads) from one wave of two CTAs per
    // SM on, 8 x 8 (256 threads) below it, where more threads per tile
    // pay; both 128 x 128 tiles.  SGEMM_GB300_FFMA_RN (8 / 16) pins it.
    const char *env_rn = std::getenv("SGEMM_GB300_FFMA_RN");
    const long long ftiles = (long long)((m + ffma::Deep::BM - 1) / ffma::Deep::BM) *
                             ((n + ffma::Deep::BN - 1) / ffma::Deep::BN) * (batch > 0 ? batch : 1);
    const bool fdeep = env_rn ? std::atoi(env_rn) == ffma::Deep::TN : ftiles >= 2LL * num_sms;
    pl->bm = fdeep ? ffma::Deep::BM : ffma::Default::BM;
    pl->bn = fdeep ? ffma::Deep::BN : ffma::Default::BN;
    pl->bk = fdeep ? ffma::Deep::BK : ffma::Default::BK;
    pl->rm = fdeep ? ffma::Deep::TM : ffma::Default::TM;
    pl->rn = fdeep ? ffma::Deep::TN : ffma::Default::TN;
    pl->threads = fdeep ? ffma::Deep::THREADS : ffma::Default::THREADS;
    pl->stages = fdeep ? ffma::Deep::STAGES : ffma::Default::STAGES;
    // rows-contiguous operands take 16-byte copies when their rows are 16-byte aligned
    pl->a_vec = op_a == SGEMM_OP_T && aligned(A, 16) && (lda % 4) == 0;
    pl->b_vec = op_b == SGEMM_OP_N && aligned(B, 16) && (ldb % 4) == 0;
    const int akind = op_a == SGEMM_OP_N ? 0 : (pl->a_vec ? 1 : 2), bkind = op_b == SGEMM_OP_T ? 0 : (pl->b_vec ? 1 : 2);
    pl->smem_bytes = fdeep ? ffma::smem_bytes<ffma::Deep>(akind, bkind) : ffma::smem_bytes<ffma::Default>(akind, bkind);
    const int tiles_m = (m + pl->bm - 1) / pl->bm;
    const int tiles_n = (n + pl->bn - 1) / pl->bn;
    pl->tiles = tiles_m * tiles_n;
    pl->grid = pl->tiles;
    pl->k_tiles = (k + pl->bk - 1) / pl->bk;
    pl->group_m = tiles_m < 8 ? tiles_m : 8;
    return SGEMM_STATUS_OK;
}

// 3-D FP32 tensor map: `nb` matrices of `rows` x `cols` (row pitch `ld`
// floats, `bstride` floats from one matrix to the next), copied in boxes of
// box_rows x box_cols of one matrix.
int make_tensor_map(CUtensorMap *map, const float *base, long long rows, long long cols, long long ld, int nb,
                    long long bstride, int box_rows, int box_cols, CUtensorMapSwizzle swizzle) {
    // a single matrix still gets a legal (16-byte multiple) batch stride
    if (nb <= 1) bstride = (rows * ld + 3) / 4 * 4;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)(nb > 1 ? nb : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)bstride * 4};
    const cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail_cuda(cudaErrorInvalidValue);
    return SGEMM_STATUS_OK;
}

// One MMA operand of the tensor-core GEMM as the kernel reads it.  `rows` is
// its extent along the tile (m for A, n for B), k its depth.
//   raw: the caller's matrix, read by TMA as stored -- kmajor: stored
//     rows x k (row pitch ld); otherwise stored k x rows (MN-major);
//   pre-split: hi / lo arrays of rows x ka per problem (pitch ka), problems
//     rows * ka apart.
//   phased: raw and K-major, but with rows TMA cannot read as one tensor:
//     read in four row phases (X on untransposed single-CTA tiles only).
struct Operand {
    bool raw = false, kmajor = true;
    bool phased = false;
    const float *hi = nullptr, *lo = nullptr;
    long long ld = 0, bstride = 0;
    int rows = 0;
};

// The operand's two tensor maps (hi / raw, and lo), boxes of box_rows of it
// by 16 k: K-major in 64-byte swizzled rows, MN-major in 32-row boxes with
// the 128-byte swizzle of 32-byte atoms (the layout the MMA reads an
// MN-major TF32 operand in).  `z` is set when the kernel should address problem
// blockIdx.y of the map (a batch of distinct matrices).
int encode_operand(const Operand &o, int k, int box_rows, int batch, CUtensorMap *hi, CUtensorMap *lo, int *z) {
    int st;
    if (o.raw) {
        const int nb = batch > 1 && o.bstride != 0 ? batch : 1;
        *z = nb > 1;
        if (o.kmajor)
            st = make_tensor_map(hi, o.hi, o.rows, k, o.ld, nb, o.bstride, box_rows, tf32x3::BK,
                                 CU_TENSOR_MAP_SWIZZLE_64B);
        else
            st = make_tensor_map(hi, o.hi, k, o.rows, o.ld, nb, o.bstride, tf32x3::BK, 32,
                                 CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B);
        if (!st) *lo = *hi;   // not read
        return st;
    }
    const long long ka = (k + 3) & ~3;
    *z = batch > 1;
    st = make_tensor_map(hi, o.hi, o.rows, k, ka, batch, (long long)o.rows * ka, box_rows, tf32x3::BK,
                         CU_TENSOR_MAP_SWIZZLE_64B);
    if (!st)
        st = make_tensor_map(lo, o.lo, o.rows, k, ka, batch, (long long)o.rows * ka, box_rows, tf32x3::BK,
                             CU_TENSOR_MAP_SWIZZLE_64B);
    return st;
}

// The four row-phase tensor maps of a phased operand (see kPhased in the
// kernel): phase j = rows j, j + 4, j + 8, ... (a row pitch of 4 * ld
// floats, a multiple of 16 bytes), based at its first row rounded down to
// 16 bytes, each row of the view extended at the front by the shift sh_j
// (0..3 floats) so that it holds k + sh_j columns: the TMA box (20 columns
// from a slab's first k, 32 row groups) then covers the slab's 16 values
// of every row, and whatever lies past k + sh_j reads as zero.  The bytes
// in front of a row (its shift) lie in the 16-byte granule of the row's
// first value.  A phase with no rows (rows < 4) repeats phase 0, whose
// values then land in tile rows that are never stored.  Its shifts go into
// *shifts (2 bits per phase).  Needs problems 16 bytes apart (bstride % 4
// == 0) in a batch.
int encode_phased(const Operand &o, int k, int batch, CUtensorMap *maps[4], int *shifts, int *z) {
    const int nb = batch > 1 && o.bstride != 0 ? batch : 1;
    *z = nb > 1;
    *shifts = 0;
    for (int j = 0; j < 4; ++j) {
        const int jj = j < o.rows ? j : 0;
        const uintptr_t first = reinterpret_cast<uintptr_t>(o.hi + (long long)jj * o.ld);
        const int sh = (int)((first & 15) / 4);
        const float *base = reinterpret_cast<const float *>(first - (first & 15));
        const long long rows_j = (o.rows - jj + 3) / 4;
        const int st = make_tensor_map(maps[j], base, rows_j, (long long)k + sh, 4 * o.ld, nb, o.bstride,
                                       tf32x3::BM / 4, tf32x3::PHASE_COLS, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st) return st;
        *shifts |= sh << (2 * j);
    }
    return SGEMM_STATUS_OK;
}

int ka_of(int k) { return (k + 3) & ~3; }

// A (m x k, lda) -> a_hi, a_lo (m x ka).
// Grids of the split kernels: about 8 blocks of 256 threads per SM, each
// looping over its share (they are HBM-bound).
constexpr int kSplitBlocks = 8 * 160;

tf32x3::SplitJob split_a_job(int m, int k, const float *A, int lda, float *a_hi, float *a_lo, int batch,
                             long long src_batch, long long dst_batch) {
    const bool vec = aligned(A, 16) && (lda % 4) == 0 && (src_batch % 4) == 0;
    const int per_row = vec ? (k / 4 > 0 ? k / 4 : 1) : k;
    int gx = (per_row + 255) / 256;
    if (gx > 16) gx = 16;
    int gy = kSplitBlocks / gx;
    if (gy < 1) gy = 1;
    if (gy > m) gy = m;
    if (gy > 65535) gy = 65535;
    // with a batch, fewer rows per problem in flight
    if (batch > 1) gy = gy / batch > 0 ? gy / batch : 1;
    return tf32x3::SplitJob{A, lda, m, k, a_hi, a_lo, ka_of(k), src_batch, dst_batch, gx, gy, vec ? 1 : 0};
}

// B (k x n, ldb) -> bt_hi, bt_lo (B^T, n x ka).
tf32x3::SplitJob split_b_job(int k, int n, const float *B, int ldb, float *bt_hi, float *bt_lo, int batch,
                             long long src_batch, long long dst_batch) {
    long long gx = (n + 63) / 64, gy = (k + 31) / 32;
    const long long budget = batch > 1 ? (kSplitBlocks / batch > 0 ? kSplitBlocks / batch : 1) : kSplitBlocks;
    if (gx > budget) gx = budget;
    if (gy > budget / gx) gy = budget / gx > 0 ? budget / gx : 1;
    return tf32x3::SplitJob{B, ldb, k, n, bt_hi, bt_lo, ka_of(k), src_batch, dst_batch, (int)gx, (int)gy, 2};
}

// Split passes in one launch (split_pair_kernel): j0, then j1 (none when j1.gx = 0).
void launch_split_pair(const tf32x3::SplitJob &j0, const tf32x3::SplitJob &j1, int batch, cudaStream_t stream) {
    const unsigned blocks = (unsigned)(j0.gx * j0.gy + j1.gx * j1.gy);
    tf32x3::split_pair_kernel<<<dim3(blocks, 1, (unsigned)batch), 256, 0, stream>>>(j0, j1);
}

int launch_split_a(int m, int k, const float *A, int lda, float *a_hi, float *a_lo, cudaStream_t stream,
                   int batch = 1, long long src_batch = 0, long long dst_batch = 0) {
    if (m == 0 || k == 0 || batch == 0) return SGEMM_STATUS_OK;
    const tf32x3::SplitJob j = split_a_job(m, k, A, lda, a_hi, a_lo, batch, src_batch, dst_batch);
    const dim3 grid(j.gx, j.gy, batch);
    if (j.kind == 1)
        tf32x3::split_a_kernel<true><<<grid, 256, 0, stream>>>(A, lda, m, k, a_hi, a_lo, j.ka, src_batch, dst_batch);
    else
        tf32x3::split_a_kernel<false><<<grid, 256, 0, stream>>>(A, lda, m, k, a_hi, a_lo, j.ka, src_batch,
                                                                dst_batch);
    return SGEMM_STATUS_OK;
}

int launch_split_b(int k, int n, const float *B, int ldb, float *bt_hi, float *bt_lo, cudaStream_t stream,
                   int batch = 1, long long src_batch = 0, long long dst_batch = 0) {
    if (n == 0 || k == 0 || batch == 0) return SGEMM_STATUS_OK;
    tf32x3::SplitJob j = split_b_job(k, n, B, ldb, bt_hi, bt_lo, batch, src_batch, dst_batch), none = j;
    none.gx = none.gy = 0;
    launch_split_pair(j, none, batch, stream);
    return SGEMM_STATUS_OK;
}

// Everything a tensor-core GEMM launch needs, prepared before anything is
// enqueued (so that a failure here leaves the stream untouched).
struct GemmLaunch {
    CUtensorMap maps[6];   // X hi, X lo, Y hi, Y lo; a phased X: phases 0..3 in 0, 1, 4, 5
    tf32x3::Params prm;
    bool xm = false, ym = false, xp = false;
};

// Builds the launch of the GEMM for operands a (m side) and b (n side):
// untransposed tiles take X = a, Y = b; TRANS tiles X = b, Y = a.
int prepare_gemm(int m, int n, int k, float alpha, const Operand &a, const Operand &b, float beta, float *C,
                 int ldc, const sgemm_plan &pl, int batch, long long stride_c, float *sk_ws, int *sk_cnt,
                 GemmLaunch *L) {
    // stream-K needs its workspace (callers that allocate nothing plan without it)
    if (pl.stream_k > 0 && (sk_ws == nullptr || sk_cnt == nullptr || batch != 1)) return SGEMM_STATUS_UNSUPPORTED;
    const Operand &x = pl.trans ? b : a, &y = pl.trans ? a : b;
    // boxes: 128 rows of X (the MMA's M, per CTA), BN rows of Y (its N;
    // half of them per CTA of a pair)
    const int y_rows = pl.trans ? pl.bm : (pl.pair ? pl.bn / 2 : pl.bn);
    tf32x3::Params &p = L->prm;
    if (y.phased || (x.phased && (pl.trans || pl.pair || !x.kmajor))) return SGEMM_STATUS_UNSUPPORTED;   // plans never ask for these
    int st;
    p.x_shift = 0;
    if (x.phased) {
        CUtensorMap *ph[4] = {&L->maps[0], &L->maps[1], &L->maps[4], &L->maps[5]};
        st = encode_phased(x, k, batch, ph, &p.x_shift, &p.x_z);
    } else {
        st = encode_operand(x, k, tf32x3::BM, batch, &L->maps[0], &L->maps[1], &p.x_z);
        if (!st) {   // not read
            L->maps[4] = L->maps[0];
            L->maps[5] = L->maps[0];
        }
    }
    if (!st) st = encode_operand(y, k, y_rows, batch, &L->maps[2], &L->maps[3], &p.y_z);
    if (st) return st;
    L->xm = x.raw && !x.kmajor;
    L->ym = y.raw && !y.kmajor;
    L->xp = x.phased;
    p.m = m;
    p.n = n;
    p.k = k;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.ldc = ldc;
    p.tiles_m = (m + pl.bm - 1) / pl.bm;
    p.tiles_n = (n + pl.bn - 1) / pl.bn;
    p.group_m = pl.group_m;
    p.stride_c = stride_c;
    p.x_src = x.phased ? tf32x3::kPhased : x.raw ? tf32x3::kRaw : tf32x3::kPreSplit;
    p.y_src = y.raw ? tf32x3::kRaw : tf32x3::kPreSplit;
    p.c_vec = pl.c_vec;
    // stream-K over stream_k CTAs, or persistent whole tiles over grid CTAs
    p.sk_ctas = pl.stream_k > 0 ? pl.stream_k : (pl.persistent ? -pl.grid : 0);
    p.sk_parts = pl.stream_k > 0 ? pl.sk_parts : 0;
    p.sk_ws = sk_ws;
    p.sk_cnt = sk_cnt;
    return SGEMM_STATUS_OK;
}

// Enqueues a prepared GEMM: clusters of split_k CTAs (consecutive in x)
// share a tile, grid y = problem.  after_split: launched right after this
// call's split pass, as its programmatic dependent, so the GEMM's set-up
// overlaps the split's tail (its producer waits for the split before the
// first load; nothing else the GEMM reads is written by it).
// SGEMM_GB300_PDL=0 turns that off.
int launch_gemm(const GemmLaunch &L, const sgemm_plan &pl, int batch, cudaStream_t stream, bool after_split) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid, (unsigned)batch, 1);
    cfg.blockDim = dim3((unsigned)tf32x3::THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)pl.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (pl.split_k > 1 || pl.pair) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = pl.pair ? 2u : (unsigned)pl.split_k;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (after_split) {
        const char *env = std::getenv("SGEMM_GB300_PDL");
        if (!(env && env[0] == '0')) {
            attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[na].val.programmaticStreamSerializationAllowed = 1;
            ++na;
        }
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    cudaError_t e;
    if (pl.pair)
        e = units::tc_pair_launch(cfg, L.xm, L.ym, L.xp, L.maps, L.prm);
    else if (pl.trans)
        e = units::tc_trans_launch(cfg, L.xm, L.ym, L.xp, L.maps, L.prm);
    else if (pl.bn == tf32x3::Narrow::BN)
        e = units::tc_narrow_launch(cfg, L.xm, L.ym, L.xp, L.maps, L.prm);
    else
        e = units::tc_wide_launch(cfg, L.xm, L.ym, L.xp, L.maps, L.prm);
    if (e != cudaSuccess) return fail_cuda(e);
    return SGEMM_STATUS_OK;
}

// Scratch of a tensor-core call (floats): the hi and lo parts of each
// operand the GEMM cannot read as stored (2 * rows * ka per problem), then
// stream-K's per-tile counters and two partial tiles per CTA.
struct Scratch {
    size_t a = 0, b = 0, sk_cnt = 0, sk_ws = 0;
    size_t total() const { return a + b + sk_cnt + sk_ws; }
};

Scratch scratch_of(int m, int n, int k, const sgemm_plan &pl, int batch) {
    Scratch sc;
    const size_t ka = (size_t)ka_of(k), cnt = (size_t)batch;
    if (!pl.a_in_kernel) sc.a = 2 * cnt * (size_t)m * ka;
    if (!pl.b_in_kernel) sc.b = 2 * cnt * (size_t)n * ka;
    if (pl.stream_k > 0) {
        sc.sk_cnt = ((size_t)pl.tiles + 3) / 4 * 4;
        sc.sk_ws = (size_t)pl.stream_k * 2 * tf32x3::BM * (pl.trans ? tf32x3::Wide::BN : pl.bn);
    }
    return sc;
}

// The tensor-core path of one call (a strided batch of `bt.count`
// problems): operands the GEMM can read as stored go to it as they are; the
// others are split into scratch first by one split_pair_kernel launch.
// `ws` is the call's scratch (scratch_of(...).total() floats), NULL when
// it needs none.  Everything is prepared before the first launch.
int run_tf32x3(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
               float *C, int ldc, const sgemm_plan &pl, cudaStream_t stream, int num_sms, const Batch &bt, float *ws) {
    const Scratch sc = scratch_of(m, n, k, pl, bt.count);
    const size_t a_elems = (size_t)m * ka_of(k), b_elems = (size_t)n * ka_of(k);
    float *a_hi = ws, *a_lo = ws + sc.a / 2, *b_hi = ws + sc.a, *b_lo = ws + sc.a + sc.b / 2;
    int *sk_cnt = pl.stream_k > 0 ? reinterpret_cast<int *>(ws + sc.a + sc.b) : nullptr;
    float *sk_ws = pl.stream_k > 0 ? ws + sc.a + sc.b + sc.sk_cnt : nullptr;
    Operand oa, ob;
    oa.rows = m;
    ob.rows = n;
    if (pl.a_in_kernel) {
        oa.raw = true;
        oa.kmajor = pl.op_a == SGEMM_OP_N;   // stored m x k; else k x m
        oa.phased = !tma_readable(A, lda, pl.op_a == SGEMM_OP_N ? m : k, bt.count, bt.sa);
        oa.hi = A;
        oa.ld = lda;
        oa.bstride = bt.sa;
    } else {
        oa.hi = a_hi;
        oa.lo = a_lo;
    }
    if (pl.b_in_kernel) {
        ob.raw = true;
        ob.kmajor = pl.op_b == SGEMM_OP_T;   // stored n x k; else k x n
        ob.hi = B;
        ob.ld = ldb;
        ob.bstride = bt.sb;
    } else {
        ob.hi = b_hi;
        ob.lo = b_lo;
    }
    GemmLaunch L;
    int st = prepare_gemm(m, n, k, alpha, oa, ob, beta, C, ldc, pl, bt.count, bt.sc, sk_ws, sk_cnt, &L);
    if (st) return st;
    cudaError_t e;
    if (sk_cnt != nullptr && (e = cudaMemsetAsync(sk_cnt, 0, (size_t)pl.tiles * sizeof(int), stream)) != cudaSuccess)
        return fail_cuda(e);
    // split pass for the operands the GEMM cannot read as stored: an operand
    // stored with k contiguous is split row by row, one stored k-major
    // through the transposing split; both in one launch
    tf32x3::SplitJob jobs[2];
    int nj = 0;
    if (!pl.a_in_kernel)
        jobs[nj++] = pl.op_a == SGEMM_OP_N ? split_a_job(m, k, A, lda, a_hi, a_lo, bt.count, bt.sa, (long long)a_elems)
                                           : split_b_job(k, m, A, lda, a_hi, a_lo, bt.count, bt.sa, (long long)a_elems);
    if (!pl.b_in_kernel)
        jobs[nj++] = pl.op_b == SGEMM_OP_N ? split_b_job(k, n, B, ldb, b_hi, b_lo, bt.count, bt.sb, (long long)b_elems)
                                           : split_a_job(n, k, B, ldb, b_hi, b_lo, bt.count, bt.sb, (long long)b_elems);
    if (nj > 0) {
        tf32x3::SplitJob none = jobs[0];
        none.gx = none.gy = 0;
        launch_split_pair(jobs[0], nj > 1 ? jobs[1] : none, bt.count, stream);
    }
    // after a split pass the GEMM starts its set-up while the split finishes
    // when it runs in one wave (measured: 2048^3 +2.4 %, 1024^3 +7 %, 512^3
    // +14 %; a many-wave GEMM gains nothing from it: 8192^3 -3 %)
    const bool pdl = nj > 0 && (long long)pl.grid * bt.count <= num_sms;
    return launch_gemm(L, pl, bt.count, stream, pdl);
}

// run_tf32x3 with the call's scratch taken from the device's stream-ordered
// pool for the duration of the call (nothing is allocated when the call
// needs no scratch).  SGEMM_GB300_FAIL_ALLOC (fault injection for tests):
// the allocation reports out-of-memory without being attempted.
int launch_tf32x3(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
                  float *C, int ldc, const sgemm_plan &pl, cudaStream_t stream, cudaMemPool_t pool, int num_sms,
                  const Batch &bt = Batch()) {
    const size_t need = scratch_of(m, n, k, pl, bt.count).total();
    float *ws = nullptr;
    if (need > 0) {
        const cudaError_t e = std::getenv("SGEMM_GB300_FAIL_ALLOC") != nullptr
                                  ? cudaErrorMemoryAllocation
                                  : cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), need * sizeof(float),
                                                            pool, stream);
        if (e != cudaSuccess) return fail_cuda(e);
    }
    const int st = run_tf32x3(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, pl, stream, num_sms, bt, ws);
    if (ws != nullptr) {
        const cudaError_t e = cudaFreeAsync(ws, stream);
        if (!st && e != cudaSuccess) return fail_cuda(e);
    }
    return st;
}

// ---------------------------------------------------------------- no-allocation variant
//
// Scratch of sgemm_tf32x3_noalloc(): a fixed array in device global memory,
// created when the module loads on a device and kept until the process
// exits.  Host code must not use the array's name as a device address (on
// the host it only names the symbol); the device address is looked up once
// per device with cudaGetSymbolAddress while that device is current.
static __device__ __align__(256) float g_noalloc_scratch[SGEMM_NOALLOC_SCRATCH_FLOATS];

std::mutex g_noalloc_mu;
float *g_noalloc_ptr[kMaxDevices] = {};

// Device address of this device's g_noalloc_scratch (looked up on first use).
int noalloc_scratch(float **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return fail_cuda(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return fail_cuda(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        g_noalloc_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return SGEMM_STATUS_OK;
}

void launch_ffma(const sgemm_plan &pl, const GemmArgs &a, int batch, cudaStream_t s) {
    const int akind = pl.op_a == SGEMM_OP_N ? 0 : (pl.a_vec ? 1 : 2);
    const int bkind = pl.op_b == SGEMM_OP_T ? 0 : (pl.b_vec ? 1 : 2);
    units::ffma_launch(pl.rn == ffma::Deep::TN, akind, bkind, a, dim3((unsigned)pl.grid, (unsigned)batch, 1), s);
}

// Status code of the bounded-wait self-test (sgemm_selftest_wait).
constexpr int kStatusSelfTest = 0x207;

// One bounded wait on an mbarrier that nothing arrives at: it runs out after
// limit_ns, records kStatusSelfTest in the status word (through the same
// mbar_wait every pipeline wait of the GEMM uses) and returns; *gave_up
// tells the host that it did.  Exercises the failure-reporting path without
// a real stall.
__global__ void selftest_wait_kernel(unsigned long long limit_ns, int *gave_up) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    *gave_up = mbar_wait(smem_u32(&bar), 0, kStatusSelfTest, limit_ns) ? 0 : 1;
}

// The bounds-check self-test: a store to element n of a buffer of n + 1
// floats whose check (i < n) fails, so a checked build skips it and records
// kStatusBounds and the check's line.  (Element n exists, so even a build
// without checks would stay inside the buffer; it is never launched there.)
__global__ void selftest_bounds_kernel(float *x, int n) {
    const int i = n;
    if (SG_IN(i < n)) x[i] = 1.f;
}

// The status words and failed-test lines of every translation unit of the
// library -- this one's split, reduction and self-test kernels, and the
// kernel units' -- read after a synchronisation: the first non-zero one of
// each in unit order (each unit keeps the first code its kernels recorded).
// `clear` resets both in every unit.
cudaError_t all_units_status(int *status, int *line, bool clear) {
    using Fn = cudaError_t (*)(int *, int *, bool);
    static const Fn fns[] = {unit_status,           units::tc_wide_status, units::tc_narrow_status,
                             units::tc_trans_status, units::tc_pair_status, units::ffma_status};
    int st = 0, ln = 0;
    for (Fn f : fns) {
        int s = 0, l = 0;
        cudaError_t e = f(&s, &l, clear);
        if (e != cudaSuccess) return e;
        if (st == 0) st = s;
        if (ln == 0) ln = l;
    }
    if (status) *status = st;
    if (line) *line = ln;
    return cudaSuccess;
}

}  // namespace

extern "C" {

int sgemm_strided_batched(int op_a, int op_b, int m, int n, int k, float alpha, const float *A, int lda,
                          long long stride_a, const float *B, int ldb, long long stride_b, float beta, float *C,
                          int ldc, long long stride_c, int batch, cudaStream_t stream, int path) {
    if (op_a != SGEMM_OP_N && op_a != SGEMM_OP_T) return 1;
    if (op_b != SGEMM_OP_N && op_b != SGEMM_OP_T) return 2;
    if (path != SGEMM_PATH_AUTO && path != SGEMM_PATH_FFMA && path != SGEMM_PATH_TF32X3)
        return SGEMM_STATUS_BAD_PATH;
    // argument positions: op_a 1, op_b 2, m 3, n 4, k 5, alpha 6, A 7, lda 8,
    // stride_a 9, B 10, ldb 11, stride_b 12, beta 13, C 14, ldc 15,
    // stride_c 16, batch 17
    if (m < 0) return 3;
    if (n < 0) return 4;
    if (k < 0) return 5;
    if (batch == 0) return SGEMM_STATUS_OK;   // an empty batch reads and writes nothing
    if (int bad = check_args(m, n, k, alpha, A, lda, B, ldb, C, ldc, op_a, op_b)) {
        static const int pos[12] = {0, 3, 4, 5, 6, 7, 8, 10, 11, 13, 14, 15};
        return pos[bad];
    }
    if (stride_a < 0) return 9;
    if (stride_b < 0) return 12;
    if (batch < 0) return 17;
    // the batch's C matrices must not overlap
    if (batch > 1 && (long long)m * n > 0 && stride_c < (long long)(m - 1) * ldc + n) return 16;
    if (m == 0 || n == 0 || batch == 0) return SGEMM_STATUS_OK;
    DeviceState *dev = nullptr;
    int st = device_state(&dev);
    if (st != SGEMM_STATUS_OK) return st;
    // grid.y carries the batch (<= 65535 per launch): larger batches go in chunks
    const long long chunk = 65535;
    for (long long b0 = 0; b0 < batch; b0 += chunk) {
        const int cnt = (int)(batch - b0 < chunk ? batch - b0 : chunk);
        const float *Ab = A ? A + b0 * stride_a : A;
        const float *Bb = B ? B + b0 * stride_b : B;
        float *Cb = C + b0 * stride_c;
        sgemm_plan pl;
        st = plan(m, n, k, alpha, Ab, lda, Bb, ldb, beta, Cb, ldc, path, dev->sms, &pl, dev->max_clusters, op_a, op_b,
                  cnt, true, stride_a, stride_b);
        if (st != SGEMM_STATUS_OK) return st;
        // 16-byte accesses need every problem's base aligned, not only the first
        if (stride_c % 4) pl.c_vec = 0;
        if (stride_a % 4) pl.a_vec = 0;
        if (stride_b % 4) pl.b_vec = 0;
        Batch bt;
        bt.count = cnt;
        bt.sa = stride_a;
        bt.sb = stride_b;
        bt.sc = stride_c;
        if (pl.kernel == kKernelScale) {
            scale_c_kernel<<<dim3(pl.grid, cnt), pl.threads, 0, stream>>>(Cb, ldc, m, n, beta, stride_c);
        } else if (pl.kernel == kKernelTf32x3) {
            if ((st = launch_tf32x3(m, n, k, alpha, Ab, lda, Bb, ldb, beta, Cb, ldc, pl, stream, dev->pool, dev->sms,
                                    bt)))
                return st;
        } else {
            GemmArgs a;
            a.m = m;
            a.n = n;
            a.k = k;
            a.alpha = alpha;
            a.beta = beta;
            a.A = Ab;
            a.lda = lda;
            a.B = Bb;
            a.ldb = ldb;
            a.C = Cb;
            a.ldc = ldc;
            a.tiles_m = (m + pl.bm - 1) / pl.bm;
            a.tiles_n = (n + pl.bn - 1) / pl.bn;
            a.group_m = pl.group_m;
            a.c_vec = pl.c_vec;
            a.stride_a = stride_a;
            a.stride_b = stride_b;
            a.stride_c = stride_c;
            launch_ffma(pl, a, cnt, stream);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail_cuda(e);
    }
    return SGEMM_STATUS_OK;
}

int sgemm_op(int op_a, int op_b, int m, int n, int k, float alpha, const float *A, int lda, const float *B,
             int ldb, float beta, float *C, int ldc, cudaStream_t stream, int path) {
    const int st = sgemm_strided_batched(op_a, op_b, m, n, k, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1,
                                         stream, path);
    // back to sgemm_op's positions (no strides)
    static const int pos[18] = {0, 1, 2, 3, 4, 5, 6, 7, 8, 0, 9, 10, 0, 11, 12, 13, 0, 0};
    return st >= 1 && st <= 17 ? pos[st] : st;
}

int sgemm_ex(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb,
             float beta, float *C, int ldc, cudaStream_t stream, int path) {
    const int st = sgemm_op(SGEMM_OP_N, SGEMM_OP_N, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, stream, path);
    return st >= 3 && st <= 13 ? st - 2 : st;   // sgemm()'s argument positions
}

int sgemm_tf32x3_split_a(int m, int k, const float *A, int lda, float *a_hi, float *a_lo, cudaStream_t stream) {
    if (m < 0) return 1;
    if (k < 0) return 2;
    const bool work = (long long)m * k > 0;
    if (work && (A == nullptr || !aligned(A, 4))) return 3;
    if (lda < imax(1, k)) return 4;
    if (work && (a_hi == nullptr || !aligned(a_hi, 16))) return 5;
    if (work && (a_lo == nullptr || !aligned(a_lo, 16))) return 6;
    if (!work) return SGEMM_STATUS_OK;
    DeviceState *dev = nullptr;
    if (int st = device_state(&dev)) return st;
    launch_split_a(m, k, A, lda, a_hi, a_lo, stream);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SGEMM_STATUS_OK : fail_cuda(e);
}

int sgemm_tf32x3_split_b(int k, int n, const float *B, int ldb, float *bt_hi, float *bt_lo, cudaStream_t stream) {
    if (k < 0) return 1;
    if (n < 0) return 2;
    const bool work = (long long)k * n > 0;
    if (work && (B == nullptr || !aligned(B, 4))) return 3;
    if (ldb < imax(1, n)) return 4;
    if (work && (bt_hi == nullptr || !aligned(bt_hi, 16))) return 5;
    if (work && (bt_lo == nullptr || !aligned(bt_lo, 16))) return 6;
    if (!work) return SGEMM_STATUS_OK;
    DeviceState *dev = nullptr;
    if (int st = device_state(&dev)) return st;
    launch_split_b(k, n, B, ldb, bt_hi, bt_lo, stream);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SGEMM_STATUS_OK : fail_cuda(e);
}

int sgemm_tf32x3_split_gemm(int m, int n, int k, float alpha, const float *a_hi, const float *a_lo,
                            const float *bt_hi, const float *bt_lo, float beta, float *C, int ldc,
                            cudaStream_t stream) {
    if (m < 0) return 1;
    if (n < 0) return 2;
    if (k < 0) return 3;
    const bool need_ab = (long long)m * n * k > 0 && alpha != 0.f;
    const float *ops[4] = {a_hi, a_lo, bt_hi, bt_lo};
    for (int i = 0; i < 4; ++i)
        if (need_ab && (ops[i] == nullptr || !aligned(ops[i], 16))) return 5 + i;
    if ((long long)m * n > 0 && (C == nullptr || !aligned(C, 4))) return 10;
    if (ldc < imax(1, n)) return 11;
    if (m == 0 || n == 0) return SGEMM_STATUS_OK;
    DeviceState *dev = nullptr;
    if (int st = device_state(&dev)) return st;
    sgemm_plan pl;
    // the plan of the tensor-core path for this shape (operand pointers only
    // matter to the FFMA path's alignment choice)
    int st = plan(m, n, k, alpha, a_hi, imax(1, k), a_hi, imax(1, n), beta, C, ldc, SGEMM_PATH_TF32X3, dev->sms, &pl,
                  dev->max_clusters, SGEMM_OP_N, SGEMM_OP_N, 1, false);   // allocates nothing: no stream-K
    if (st) return st;
    pl.a_in_kernel = 0;   // the operands are split already
    pl.b_in_kernel = 0;
    if (pl.kernel == kKernelScale) {
        scale_c_kernel<<<pl.grid, pl.threads, 0, stream>>>(C, ldc, m, n, beta, 0);
    } else {
        Operand oa, ob;
        oa.rows = m;
        oa.hi = a_hi;
        oa.lo = a_lo;
        ob.rows = n;
        ob.hi = bt_hi;
        ob.lo = bt_lo;
        GemmLaunch L;
        if ((st = prepare_gemm(m, n, k, alpha, oa, ob, beta, C, ldc, pl, 1, 0, nullptr, nullptr, &L))) return st;
        if ((st = launch_gemm(L, pl, 1, stream, false))) return st;
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SGEMM_STATUS_OK : fail_cuda(e);
}

int sgemm_tf32x3_noalloc(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb,
                         float beta, float *C, int ldc, cudaStream_t stream) {
    if (int bad = check_args(m, n, k, alpha, A, lda, B, ldb, C, ldc)) return bad;
    if (m == 0 || n == 0) return SGEMM_STATUS_OK;
    DeviceState *dev = nullptr;
    int st = device_state(&dev);
    if (st != SGEMM_STATUS_OK) return st;
    sgemm_plan pl;
    st = plan(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, SGEMM_PATH_TF32X3, dev->sms, &pl, dev->max_clusters,
              SGEMM_OP_N, SGEMM_OP_N, 1, false);   // no stream-K workspace in the fixed scratch
    if (st != SGEMM_STATUS_OK) return st;
    // read every operand TMA can read as stored, whatever the size (the
    // plan splits a large B with the split pass, which is faster there):
    // scratch only for a B whose rows TMA cannot read, and for such an A on
    // transposed tiles (elsewhere the GEMM reads it in row phases).  With
    // both read by TMA as stored, large problems run on CTA pairs, which
    // split B in half the shared-memory traffic per SM (measured, whole
    // call: 8192^3 4.29 ms against 5.8 ms on single-CTA 128 x 256 tiles);
    // pairs take no phased A
    if (pl.kernel != kKernelScale && tma_readable(B, ldb, k, 1, 0)) {
        pl.b_in_kernel = 1;
        if (pl.a_in_kernel && tma_readable(A, lda, m, 1, 0) && !pl.trans && (long long)m * n * k > (1LL << 31))
            set_pair_plan(m, n, k, &pl);
    }
    if (pl.kernel == kKernelScale) {
        scale_c_kernel<<<pl.grid, pl.threads, 0, stream>>>(C, ldc, m, n, beta, 0);
    } else {
        // only operands the GEMM cannot read as stored need scratch: their
        // split parts go into the fixed array instead of the pool
        const size_t need = scratch_of(m, n, k, pl, 1).total();
        if (need > (size_t)SGEMM_NOALLOC_SCRATCH_FLOATS) return SGEMM_STATUS_TOO_LARGE;
        float *ws = nullptr;
        if (need > 0 && (st = noalloc_scratch(&ws))) return st;
        // the split pass writes every element the GEMM reads, so nothing
        // left in the array by an earlier call is ever used
        if ((st = run_tf32x3(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, pl, stream, dev->sms, Batch(), ws)))
            return st;
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SGEMM_STATUS_OK : fail_cuda(e);
}

int sgemm(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
          float *C, int ldc, cudaStream_t stream) {
    return sgemm_ex(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, stream, SGEMM_PATH_AUTO);
}

int sgemm_plan_for(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb,
                   float beta, const float *C, int ldc, int path, int num_sms, sgemm_plan *out) {
    if (out == nullptr) return SGEMM_STATUS_UNSUPPORTED;
    if (num_sms == 0) {   // the current device, as a call would plan it
        DeviceState *dev = nullptr;
        if (int st = device_state(&dev)) return st;
        return plan(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, path, dev->sms, out, dev->max_clusters);
    }
    return plan(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, path, num_sms, out);
}

int reduce_sum_f32(const float *x, long long n, float *out, cudaStream_t stream) {
    if (n < 0) return 2;
    if (n > 0 && (x == nullptr || !aligned(x, 4))) return 1;
    if (out == nullptr || !aligned(out, 4)) return 3;
    DeviceState *dev = nullptr;
    if (int st = device_state(&dev)) return st;
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), stream);
    if (e != cudaSuccess) return fail_cuda(e);
    if (n > 0) {
        long long blocks = (n + 4LL * reduce::THREADS * 4 - 1) / (4LL * reduce::THREADS * 4);
        const long long cap = (long long)dev->sms * reduce::BLOCKS_PER_SM;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        if (aligned(x, 16))
            reduce::reduce_sum_kernel<true><<<(unsigned)blocks, reduce::THREADS, 0, stream>>>(x, n, out);
        else
            reduce::reduce_sum_kernel<false><<<(unsigned)blocks, reduce::THREADS, 0, stream>>>(x, n, out);
        e = cudaGetLastError();
        if (e != cudaSuccess) return fail_cuda(e);
    }
    return SGEMM_STATUS_OK;
}

const char *sgemm_status_string(int status) {
    // Argument errors name the 1-based position in the call that returned
    // them; the entry points number their arguments differently (the header
    // lists each one's positions), so the text names only the position.
    static const char *const kArg[18] = {
        "success",
        "invalid argument 1 (1-based position in the call's argument list)",
        "invalid argument 2 (1-based position in the call's argument list)",
        "invalid argument 3 (1-based position in the call's argument list)",
        "invalid argument 4 (1-based position in the call's argument list)",
        "invalid argument 5 (1-based position in the call's argument list)",
        "invalid argument 6 (1-based position in the call's argument list)",
        "invalid argument 7 (1-based position in the call's argument list)",
        "invalid argument 8 (1-based position in the call's argument list)",
        "invalid argument 9 (1-based position in the call's argument list)",
        "invalid argument 10 (1-based position in the call's argument list)",
        "invalid argument 11 (1-based position in the call's argument list)",
        "invalid argument 12 (1-based position in the call's argument list)",
        "invalid argument 13 (1-based position in the call's argument list)",
        "invalid argument 14 (1-based position in the call's argument list)",
        "invalid argument 15 (1-based position in the call's argument list)",
        "invalid argument 16 (1-based position in the call's argument list)",
        "invalid argument 17 (1-based position in the call's argument list)",
    };
    if (status >= 0 && status <= 17) return kArg[status];
    switch (status) {
        case SGEMM_STATUS_TOO_LARGE:
            return "problem too large for the fixed no-allocation scratch (SGEMM_NOALLOC_SCRATCH_FLOATS)";
        case SGEMM_STATUS_BAD_PATH: return "unknown kernel path";
        case SGEMM_STATUS_UNSUPPORTED: return "unsupported request (no plan structure given, or a checked-build-only call)";
        case SGEMM_STATUS_CUDA_ERROR: return "CUDA runtime error (see sgemm_last_cuda_error)";
        default: return "unknown status";
    }
}

int sgemm_last_cuda_error(void) { return g_last_cuda_error; }

int sgemm_device_status(int *flag, int clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e);
    int v = 0;
    if ((e = all_units_status(&v, nullptr, clear != 0)) != cudaSuccess) return fail_cuda(e);
    if (flag) *flag = v;
    return SGEMM_STATUS_OK;
}

int sgemm_selftest_wait(unsigned long long limit_ns, int *gave_up) {
    if (limit_ns == 0 || limit_ns > 10000000000ull) return 1;
    if (gave_up == nullptr) return 2;
    int *d = nullptr;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&d), sizeof(int));
    if (e != cudaSuccess) return fail_cuda(e);
    selftest_wait_kernel<<<1, 32>>>(limit_ns, d);
    if ((e = cudaGetLastError()) == cudaSuccess) e = cudaDeviceSynchronize();
    int v = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&v, d, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(d);
    if (e != cudaSuccess) return fail_cuda(e);
    *gave_up = v;
    return SGEMM_STATUS_OK;
}

int sgemm_bounds_line(int *line, int clear) {
    if (line == nullptr) return 1;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e);
    int v = 0;
    if ((e = all_units_status(nullptr, &v, clear != 0)) != cudaSuccess) return fail_cuda(e);
    *line = v;
    return SGEMM_STATUS_OK;
}

int sgemm_selftest_bounds(int *line) {
#ifndef SGEMM_GB300_CHECKED
    (void)line;
    return SGEMM_STATUS_UNSUPPORTED;
#else
    if (line == nullptr) return 1;
    constexpr int n = 32;
    float *d = nullptr;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&d), (n + 1) * sizeof(float));
    if (e != cudaSuccess) return fail_cuda(e);
    selftest_bounds_kernel<<<1, 1>>>(d, n);
    if ((e = cudaGetLastError()) == cudaSuccess) e = cudaDeviceSynchronize();
    int v = 0;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_sgemm_bad_line, sizeof(int));
    cudaFree(d);
    if (e != cudaSuccess) return fail_cuda(e);
    *line = v;
    return SGEMM_STATUS_OK;
#endif
}

#ifdef SGEMM_GB300_CHECKED
const char *sgemm_version(void) { return "sgemm_gb300 0.1 (sm_103a, checked)"; }
#else
const char *sgemm_version(void) { return "sgemm_gb300 0.1 (sm_103a)"; }
#endif

}  // extern "C"
