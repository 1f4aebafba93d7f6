// Kernels for bits = 2, group_size = 64.
#include "qmv_launch.cuh"

namespace qmv {
cudaError_t launch_b2g64(int V, int R, const CUtensorMap &map, const Params &p, dim3 grid, int threads,
                          size_t smem, cudaStream_t stream)
{
    return launch_bits_gs<2, 64>(V, R, map, p, grid, threads, smem, stream);
}
}  // namespace qmv
