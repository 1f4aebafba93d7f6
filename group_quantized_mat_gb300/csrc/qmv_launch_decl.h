// Entry points of the per-(bits, group_size) kernel tables (qmv_inst_*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "qmv_plan.h"

namespace qmv {

// Warps per CTA of the kernel for V vectors (its launch bounds): consumer
// warps, then producer warps.
inline int consumer_warps(int V) { return V == 1 ? 16 : 10; }
inline int producer_warps(int V) { return V == 1 ? 4 : 2; }

struct Launch {
    dim3 grid;
    int threads;
    size_t smem;
    bool pdl;  // launch with a programmatic dependency on the preceding grid
};

#define QMV_DECLARE_LAUNCH(name) \
    cudaError_t name(int V, const CUtensorMap &map_s, const CUtensorMap &map_b, const Params &p, const Launch &l, \
                     cudaStream_t stream);
QMV_DECLARE_LAUNCH(launch_b4g64)
QMV_DECLARE_LAUNCH(launch_b4g128)
QMV_DECLARE_LAUNCH(launch_b2g64)
QMV_DECLARE_LAUNCH(launch_b2g128)
#undef QMV_DECLARE_LAUNCH

}  // namespace qmv
