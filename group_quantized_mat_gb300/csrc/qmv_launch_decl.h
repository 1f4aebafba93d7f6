// Entry points of the per-(bits, group_size) kernel tables (qmv_inst_*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "qmv_plan.h"

namespace qmv {

// Warps a CTA may have for this V (the kernels' launch bounds).
inline int max_warps(int V) { return V == 1 ? 16 : 8; }

#define QMV_DECLARE_LAUNCH(name)                                                                            \
    cudaError_t name(int V, int R, const CUtensorMap &map, const Params &p, dim3 grid, int threads, \
                     size_t smem, cudaStream_t stream);
QMV_DECLARE_LAUNCH(launch_b4g64)
QMV_DECLARE_LAUNCH(launch_b4g128)
QMV_DECLARE_LAUNCH(launch_b2g64)
QMV_DECLARE_LAUNCH(launch_b2g128)
#undef QMV_DECLARE_LAUNCH

}  // namespace qmv
