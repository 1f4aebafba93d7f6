// Kernels for bits = 4, group_size = 128.
#include "qmv_launch.cuh"

namespace qmv {
cudaError_t launch_b4g128(int V, const CUtensorMap &map, const Params &p, int grid_y, size_t smem,
                           cudaStream_t stream)
{
    return launch_bits_gs<4, 128>(V, map, p, grid_y, smem, stream);
}
}  // namespace qmv
