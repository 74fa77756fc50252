// Tensor-core GEMM instances on 128 x 128 tiles: kernel attributes, cluster
// capacity and launches (a unit of its own: see units.h).
#include "tc_units.cuh"

namespace sgemm_gb300 {
namespace units {

cudaError_t tc_narrow_attrs() { return set_tc_attr<tf32x3::Narrow, false>(); }
cudaError_t tc_narrow_clusters(int S, int *out) { return max_clusters_of<tf32x3::Narrow>(S, out); }
cudaError_t tc_narrow_launch(const cudaLaunchConfig_t &cfg, bool xm, bool ym, bool xp, const CUtensorMap *maps,
                              const tf32x3::Params &p) {
    return launch_tc<tf32x3::Narrow, false>(cfg, xm, ym, xp, maps, p);
}
cudaError_t tc_narrow_status(int *status, int *line, bool clear) { return unit_status(status, line, clear); }

}  // namespace units
}  // namespace sgemm_gb300
