// Launch helpers of the tensor-core GEMM kernel, instantiated by the unit
// that includes this file for its own tile configuration.
#pragma once
#include "units.h"

namespace sgemm_gb300 {
namespace units {

template <class Cfg, bool TRANS, bool XM, bool YM, bool XP = false>
cudaError_t set_tc_attr_one() {
    return cudaFuncSetAttribute(tf32x3::tf32x3_gemm_kernel<Cfg, TRANS, XM, YM, XP>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
}

// The four operand-layout variants of one tile shape (X and Y each K-major
// or MN-major), and on untransposed single-CTA tiles the two with X read in
// row phases.
template <class Cfg, bool TRANS>
cudaError_t set_tc_attr() {
    cudaError_t e = set_tc_attr_one<Cfg, TRANS, false, false>();
    if (e == cudaSuccess) e = set_tc_attr_one<Cfg, TRANS, false, true>();
    if (e == cudaSuccess) e = set_tc_attr_one<Cfg, TRANS, true, false>();
    if (e == cudaSuccess) e = set_tc_attr_one<Cfg, TRANS, true, true>();
    if constexpr (!TRANS && !Cfg::PAIR) {
        if (e == cudaSuccess) e = set_tc_attr_one<Cfg, false, false, false, true>();
        if (e == cudaSuccess) e = set_tc_attr_one<Cfg, false, false, true, true>();
    }
    return e;
}

// Clusters of S CTAs of the tensor-core kernel that can be resident at once
// (thread-block clusters cannot span GPCs, so this is below sms / S).
template <class Cfg>
cudaError_t max_clusters_of(int S, int *out) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(S * 64), 1, 1);
    cfg.blockDim = dim3((unsigned)tf32x3::THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)Cfg::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    *out = 0;
    return cudaOccupancyMaxActiveClusters(out, tf32x3::tf32x3_gemm_kernel<Cfg, false, false, true>, &cfg);
}

template <class Cfg, bool TRANS, bool XM, bool YM, bool XP = false>
cudaError_t launch_tc_one(const cudaLaunchConfig_t &cfg, const CUtensorMap *maps, const tf32x3::Params &a) {
    return cudaLaunchKernelEx(&cfg, tf32x3::tf32x3_gemm_kernel<Cfg, TRANS, XM, YM, XP>, maps[0], maps[1], maps[2],
                              maps[3], maps[4], maps[5], a);
}

// xm / ym: X / Y read MN-major; xp: X read in row phases (untransposed
// single-CTA tiles only; prepare_gemm rejects the rest)
template <class Cfg, bool TRANS>
cudaError_t launch_tc(const cudaLaunchConfig_t &cfg, bool xm, bool ym, bool xp, const CUtensorMap *maps,
                      const tf32x3::Params &a) {
    if constexpr (!TRANS && !Cfg::PAIR) {
        if (xp) return ym ? launch_tc_one<Cfg, false, false, true, true>(cfg, maps, a)
                          : launch_tc_one<Cfg, false, false, false, true>(cfg, maps, a);
    }
    if (xm) return ym ? launch_tc_one<Cfg, TRANS, true, true>(cfg, maps, a) : launch_tc_one<Cfg, TRANS, true, false>(cfg, maps, a);
    return ym ? launch_tc_one<Cfg, TRANS, false, true>(cfg, maps, a) : launch_tc_one<Cfg, TRANS, false, false>(cfg, maps, a);
}

}  // namespace units
}  // namespace sgemm_gb300
