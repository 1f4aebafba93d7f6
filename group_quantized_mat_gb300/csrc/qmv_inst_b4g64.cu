// Kernels for bits = 4, group_size = 64.
#include "qmv_launch.cuh"

namespace qmv {
cudaError_t launch_b4g64(int V, const CUtensorMap &map_s, const CUtensorMap &map_b, const Params &p, const Launch &l,
                         cudaStream_t stream)
{
    return launch_bits_gs<4, 64>(V, map_s, map_b, p, l, stream);
}
}  // namespace qmv
