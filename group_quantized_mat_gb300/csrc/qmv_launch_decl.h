// Entry points of the per-(bits, group_size) kernel tables (qmv_inst_*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "qmv_plan.h"

namespace qmv {

cudaError_t launch_b4g64(int V, const CUtensorMap &map, const Params &p, int grid_y, size_t smem,
                         cudaStream_t stream);
cudaError_t launch_b4g128(int V, const CUtensorMap &map, const Params &p, int grid_y, size_t smem,
                          cudaStream_t stream);
cudaError_t launch_b2g64(int V, const CUtensorMap &map, const Params &p, int grid_y, size_t smem,
                         cudaStream_t stream);
cudaError_t launch_b2g128(int V, const CUtensorMap &map, const Params &p, int grid_y, size_t smem,
                          cudaStream_t stream);

}  // namespace qmv
