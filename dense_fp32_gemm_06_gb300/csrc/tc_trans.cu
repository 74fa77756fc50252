// Tensor-core GEMM instances on transposed 256 x 128 tiles (C^T = B^T A^T,
// n <= 128): kernel attributes and launches (a unit of its own: see
// units.h).  Their cluster capacity is the 128 x 256 unit's (the same
// threads and shared memory), so this unit reports none.
#include "tc_units.cuh"

namespace sgemm_gb300 {
namespace units {

cudaError_t tc_trans_attrs() { return set_tc_attr<tf32x3::Wide, true>(); }
cudaError_t tc_trans_clusters(int, int *out) {
    *out = 0;
    return cudaSuccess;
}
cudaError_t tc_trans_launch(const cudaLaunchConfig_t &cfg, bool xm, bool ym, bool xp, const CUtensorMap *maps,
                            const tf32x3::Params &p) {
    return launch_tc<tf32x3::Wide, true>(cfg, xm, ym, xp, maps, p);
}
cudaError_t tc_trans_status(int *status, int *line, bool clear) { return unit_status(status, line, clear); }

}  // namespace units
}  // namespace sgemm_gb300
