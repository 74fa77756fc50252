// Sum of an FP32 array, s = sum_i x_i, on sm_103a.
//
// The block reduction of aerisun.top "GPU 访存与计算优化" (section "Reduce 的
// 分层归约"): each thread first accumulates its share of the array in
// registers (grid-stride loop), a warp then combines its 32 values with
// shuffles, the warps' results meet in shared memory and the first warp
// combines them, and one atomic add per block commits the block's sum.  On
// GB300 the loop reads float4 where the array is 16-byte aligned and keeps
// four independent accumulators per thread, so each thread has several
// 16-byte loads in flight (the bytes-in-flight = bandwidth x latency
// requirement of the same page's Little's-law section); the grid is a few
// blocks per SM.  The block commit order is not fixed, so the last bits of
// the result may vary between runs (the page's own note on summation order).
#pragma once
#include <cstdint>

#include "ptx.cuh"

#include "../../include/sgemm_gb300.h"

namespace sgemm_gb300 {
namespace reduce {

// the launch shape the header states (its error bound depends on it)
constexpr int THREADS = SGEMM_REDUCE_THREADS;
constexpr int WARPS = THREADS / 32;
constexpr int BLOCKS_PER_SM = SGEMM_REDUCE_BLOCKS_PER_SM;
static_assert(WARPS <= 32, "one warp combines the block's warp sums");

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
    return v;
}

// *out must be zero (or a running total) before the launch.
template <bool VEC>
__global__ void __launch_bounds__(THREADS) reduce_sum_kernel(const float *__restrict__ x, long long n,
                                                             float *__restrict__ out) {
    const long long gtid = (long long)blockIdx.x * THREADS + threadIdx.x;
    const long long gstride = (long long)gridDim.x * THREADS;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    long long tail = 0;
    if constexpr (VEC) {
        const long long n4 = n / 4;
        const float4 *x4 = reinterpret_cast<const float4 *>(x);
        long long i = gtid;
        for (; i + gstride < n4; i += 2 * gstride) {
            if (!SG_IN(i >= 0 && 4 * (i + gstride) + 4 <= n)) continue;
            const float4 u = __ldg(x4 + i), v = __ldg(x4 + i + gstride);
            a0 += u.x;
            a1 += u.y;
            a2 += u.z;
            a3 += u.w;
            a0 += v.x;
            a1 += v.y;
            a2 += v.z;
            a3 += v.w;
        }
        if (i < n4 && SG_IN(4 * i + 4 <= n)) {
            const float4 u = __ldg(x4 + i);
            a0 += u.x;
            a1 += u.y;
            a2 += u.z;
            a3 += u.w;
        }
        tail = 4 * n4;
    }
    for (long long i = tail + gtid; i < n; i += gstride)
        if (SG_IN(i >= 0)) a0 += __ldg(x + i);
    float v = warp_sum((a0 + a1) + (a2 + a3));
    __shared__ float partial[WARPS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0 && SG_IN(warp < WARPS)) partial[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = warp_sum(lane < WARPS ? partial[lane] : 0.f);
        if (lane == 0) atomicAdd(out, v);
    }
}

}  // namespace reduce
}  // namespace sgemm_gb300
