// FFMA GEMM instances (both tile configurations, every loader
// combination): kernel attributes and launches (a unit of its own: see
// units.h).
#include "units.h"

namespace sgemm_gb300 {
namespace units {
namespace {

template <class Cfg, class AL, class BL>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(ffma::ffma_sgemm_kernel<Cfg, AL, BL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                ffma::Layout<Cfg, AL, BL>::SMEM_BYTES);
}

template <class Cfg, class AL>
cudaError_t set_attr_all_b() {
    using L = ffma::Loaders<Cfg>;
    cudaError_t e = set_attr<Cfg, AL, typename L::BScatter>();
    if (e == cudaSuccess) e = set_attr<Cfg, AL, typename L::BVec>();
    if (e == cudaSuccess) e = set_attr<Cfg, AL, typename L::BScalar>();
    return e;
}

template <class Cfg>
cudaError_t set_attr_all() {
    using L = ffma::Loaders<Cfg>;
    cudaError_t e = set_attr_all_b<Cfg, typename L::AScatter>();
    if (e == cudaSuccess) e = set_attr_all_b<Cfg, typename L::AVec>();
    if (e == cudaSuccess) e = set_attr_all_b<Cfg, typename L::AScalar>();
    return e;
}

template <class Cfg, class AL, class BL>
void launch_t(const GemmArgs &a, dim3 grid, cudaStream_t s) {
    ffma::ffma_sgemm_kernel<Cfg, AL, BL><<<grid, Cfg::THREADS, ffma::Layout<Cfg, AL, BL>::SMEM_BYTES, s>>>(a);
}

template <class Cfg, class AL>
void launch_b(int bkind, const GemmArgs &a, dim3 grid, cudaStream_t s) {
    using L = ffma::Loaders<Cfg>;
    if (bkind == 0) launch_t<Cfg, AL, typename L::BScatter>(a, grid, s);
    else if (bkind == 1) launch_t<Cfg, AL, typename L::BVec>(a, grid, s);
    else launch_t<Cfg, AL, typename L::BScalar>(a, grid, s);
}

template <class Cfg>
void launch_cfg(int akind, int bkind, const GemmArgs &a, dim3 grid, cudaStream_t s) {
    using L = ffma::Loaders<Cfg>;
    if (akind == 0) launch_b<Cfg, typename L::AScatter>(bkind, a, grid, s);
    else if (akind == 1) launch_b<Cfg, typename L::AVec>(bkind, a, grid, s);
    else launch_b<Cfg, typename L::AScalar>(bkind, a, grid, s);
}

}  // namespace

cudaError_t ffma_attrs() {
    cudaError_t e = set_attr_all<ffma::Default>();
    if (e == cudaSuccess) e = set_attr_all<ffma::Deep>();
    return e;
}

void ffma_launch(bool deep, int akind, int bkind, const GemmArgs &a, dim3 grid, cudaStream_t s) {
    if (deep)
        launch_cfg<ffma::Deep>(akind, bkind, a, grid, s);
    else
        launch_cfg<ffma::Default>(akind, bkind, a, grid, s);
}

cudaError_t ffma_status(int *status, int *line, bool clear) { return unit_status(status, line, clear); }

}  // namespace units
}  // namespace sgemm_gb300
