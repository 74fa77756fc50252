// C ABI of the GB300 SGEMM library: argument checks, launch planning and
// kernel launches.  Declared in include/sgemm_gb300.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/sgemm_gb300.h"
#include "ffma_sgemm.cuh"

using namespace sgemm_gb300;

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int sms = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

// Kernel ids in sgemm_plan::kernel.
constexpr int kKernelFfmaCpAsync = 0;
constexpr int kKernelScale = 1;
constexpr int kKernelFfmaTma = 2;

int fail_cuda(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return SGEMM_STATUS_CUDA_ERROR;
}

template <bool BV, bool CV>
cudaError_t set_ffma_attr() {
    return cudaFuncSetAttribute(ffma::ffma_sgemm_kernel<ffma::Default, BV, CV>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, ffma::Default::SMEM_BYTES);
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
        if ((e = set_ffma_attr<true, true>()) != cudaSuccess) return fail_cuda(e);
        if ((e = set_ffma_attr<true, false>()) != cudaSuccess) return fail_cuda(e);
        if ((e = set_ffma_attr<false, true>()) != cudaSuccess) return fail_cuda(e);
        if ((e = set_ffma_attr<false, false>()) != cudaSuccess) return fail_cuda(e);
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

// BLAS-style argument check; returns the 1-based position of the first bad
// argument, or 0.
int check_args(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb,
               const float *C, int ldc) {
    if (m < 0) return 1;
    if (n < 0) return 2;
    if (k < 0) return 3;
    const bool need_ab = (long long)m * n * k > 0 && alpha != 0.f;
    if (need_ab && (A == nullptr || !aligned(A, 4))) return 5;
    if (lda < imax(1, k)) return 6;
    if (need_ab && (B == nullptr || !aligned(B, 4))) return 7;
    if (ldb < imax(1, n)) return 8;
    if ((long long)m * n > 0 && (C == nullptr || !aligned(C, 4))) return 10;
    if (ldc < imax(1, n)) return 11;
    return 0;
}

bool tma_ok(const void *p, int ld) { return aligned(p, 16) && (ld % 4) == 0; }

int plan(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
         const float *C, int ldc, int path, int num_sms, sgemm_plan *pl) {
    (void)beta;
    std::memset(pl, 0, sizeof(*pl));
    if (path != SGEMM_PATH_AUTO && path != SGEMM_PATH_FFMA && path != SGEMM_PATH_TF32X3)
        return SGEMM_STATUS_BAD_PATH;
    if (int bad = check_args(m, n, k, alpha, A, lda, B, ldb, C, ldc)) return bad;
    if (m == 0 || n == 0) return SGEMM_STATUS_OK;
    if (path == SGEMM_PATH_TF32X3) return SGEMM_STATUS_UNSUPPORTED;
    if (num_sms <= 0) num_sms = 1;
    pl->path = SGEMM_PATH_FFMA;
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
    pl->kernel = kKernelFfmaCpAsync;
    pl->bm = ffma::Default::BM;
    pl->bn = ffma::Default::BN;
    pl->bk = ffma::Default::BK;
    pl->rm = ffma::Default::TM;
    pl->rn = ffma::Default::TN;
    pl->threads = ffma::Default::THREADS;
    pl->stages = ffma::Default::STAGES;
    pl->smem_bytes = ffma::Default::SMEM_BYTES;
    pl->b_vec = aligned(B, 16) && (ldb % 4) == 0;
    const int tiles_m = (m + pl->bm - 1) / pl->bm;
    const int tiles_n = (n + pl->bn - 1) / pl->bn;
    pl->tiles = tiles_m * tiles_n;
    pl->grid = pl->tiles;
    pl->k_tiles = (k + pl->bk - 1) / pl->bk;
    pl->group_m = tiles_m < 8 ? tiles_m : 8;
    return SGEMM_STATUS_OK;
}

// 2-D row-major FP32 tensor map: `rows` x `cols` with a row pitch of `ld`
// floats, copied in boxes of box_rows x box_cols.
int make_tensor_map(CUtensorMap *map, const float *base, int rows, int cols, int ld, int box_rows, int box_cols,
                    CUtensorMapSwizzle swizzle) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail_cuda(cudaErrorInvalidValue);
    return SGEMM_STATUS_OK;
}

template <bool BV, bool CV>
void launch_ffma(const GemmArgs &a, const sgemm_plan &pl, cudaStream_t s) {
    ffma::ffma_sgemm_kernel<ffma::Default, BV, CV><<<pl.grid, pl.threads, pl.smem_bytes, s>>>(a);
}

}  // namespace

extern "C" {

int sgemm_ex(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb,
             float beta, float *C, int ldc, cudaStream_t stream, int path) {
    if (path != SGEMM_PATH_AUTO && path != SGEMM_PATH_FFMA && path != SGEMM_PATH_TF32X3)
        return SGEMM_STATUS_BAD_PATH;
    if (int bad = check_args(m, n, k, alpha, A, lda, B, ldb, C, ldc)) return bad;
    if (m == 0 || n == 0) return SGEMM_STATUS_OK;
    DeviceState *dev = nullptr;
    int st = device_state(&dev);
    if (st != SGEMM_STATUS_OK) return st;
    sgemm_plan pl;
    st = plan(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, path, dev->sms, &pl);
    if (st != SGEMM_STATUS_OK) return st;
    if (pl.kernel == kKernelScale) {
        scale_c_kernel<<<pl.grid, pl.threads, 0, stream>>>(C, ldc, m, n, beta);
    } else {
        GemmArgs a;
        a.m = m;
        a.n = n;
        a.k = k;
        a.alpha = alpha;
        a.beta = beta;
        a.A = A;
        a.lda = lda;
        a.B = B;
        a.ldb = ldb;
        a.C = C;
        a.ldc = ldc;
        a.tiles_m = (m + pl.bm - 1) / pl.bm;
        a.tiles_n = (n + pl.bn - 1) / pl.bn;
        a.group_m = pl.group_m;
        if (pl.b_vec) {
            if (pl.c_vec) launch_ffma<true, true>(a, pl, stream);
            else launch_ffma<true, false>(a, pl, stream);
        } else {
            if (pl.c_vec) launch_ffma<false, true>(a, pl, stream);
            else launch_ffma<false, false>(a, pl, stream);
        }
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e);
    return SGEMM_STATUS_OK;
}

int sgemm(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
          float *C, int ldc, cudaStream_t stream) {
    return sgemm_ex(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, stream, SGEMM_PATH_AUTO);
}

int sgemm_plan_for(int m, int n, int k, float alpha, const float *A, int lda, const float *B, int ldb,
                   float beta, const float *C, int ldc, int path, int num_sms, sgemm_plan *out) {
    if (out == nullptr) return SGEMM_STATUS_UNSUPPORTED;
    return plan(m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, path, num_sms, out);
}

const char *sgemm_status_string(int status) {
    switch (status) {
        case SGEMM_STATUS_OK: return "success";
        case 1: return "invalid argument 1: m < 0";
        case 2: return "invalid argument 2: n < 0";
        case 3: return "invalid argument 3: k < 0";
        case 5: return "invalid argument 5: A is NULL or not 4-byte aligned";
        case 6: return "invalid argument 6: lda < max(1, k)";
        case 7: return "invalid argument 7: B is NULL or not 4-byte aligned";
        case 8: return "invalid argument 8: ldb < max(1, n)";
        case 10: return "invalid argument 10: C is NULL or not 4-byte aligned";
        case 11: return "invalid argument 11: ldc < max(1, n)";
        case SGEMM_STATUS_BAD_PATH: return "unknown kernel path";
        case SGEMM_STATUS_UNSUPPORTED: return "the requested path cannot run this problem";
        case SGEMM_STATUS_CUDA_ERROR: return "CUDA runtime error (see sgemm_last_cuda_error)";
        default: return "unknown status";
    }
}

int sgemm_last_cuda_error(void) { return g_last_cuda_error; }

int sgemm_device_status(int *flag, int clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e);
    int v = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_sgemm_status, sizeof(int))) != cudaSuccess) return fail_cuda(e);
    if (flag) *flag = v;
    if (clear) {
        const int zero = 0;
        if ((e = cudaMemcpyToSymbol(g_sgemm_status, &zero, sizeof(int))) != cudaSuccess) return fail_cuda(e);
    }
    return SGEMM_STATUS_OK;
}

const char *sgemm_version(void) { return "sgemm_gb300 0.1 (sm_103a)"; }

}  // extern "C"
