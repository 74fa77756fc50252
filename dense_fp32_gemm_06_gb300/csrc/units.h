// Host entry points of the library's kernel translation units.  Each unit
// (tc_wide.cu, tc_narrow.cu, tc_trans.cu, tc_pair.cu, ffma.cu) compiles its
// own kernel instances -- so that the units build in parallel -- and keeps
// its own device status word; sgemm_api.cu reaches them through these.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "ffma_sgemm.cuh"
#include "tf32x3_sgemm.cuh"

namespace sgemm_gb300 {
namespace units {

// The tensor-core units, one per tile configuration: 128 x 256 (Wide),
// 128 x 128 (Narrow), transposed 256 x 128 (Wide, TRANS) and CTA pairs.
// attrs: sets every instance's shared-memory limit; clusters: how many
// clusters of S CTAs fit at once (not for the transposed unit); launch: the
// instance for the operand layouts xm / ym (MN-major X / Y) and xp (X in row
// phases); status: the unit's status word and failed-test line.
#define SG_TC_UNIT_DECL(name)                                                                                      \
    cudaError_t tc_##name##_attrs();                                                                              \
    cudaError_t tc_##name##_clusters(int S, int *out);                                                           \
    cudaError_t tc_##name##_launch(const cudaLaunchConfig_t &cfg, bool xm, bool ym, bool xp, const CUtensorMap *maps, \
                                   const tf32x3::Params &p);                                                    \
    cudaError_t tc_##name##_status(int *status, int *line, bool clear);
SG_TC_UNIT_DECL(wide)
SG_TC_UNIT_DECL(narrow)
SG_TC_UNIT_DECL(trans)
SG_TC_UNIT_DECL(pair)
#undef SG_TC_UNIT_DECL

// The FFMA unit: both configurations (deep: 8 x 16 per thread), every
// loader combination (akind, bkind: 0 scatter, 1 direct 16-byte, 2 direct
// 4-byte).
cudaError_t ffma_attrs();
void ffma_launch(bool deep, int akind, int bkind, const GemmArgs &a, dim3 grid, cudaStream_t s);
cudaError_t ffma_status(int *status, int *line, bool clear);

}  // namespace units
}  // namespace sgemm_gb300
