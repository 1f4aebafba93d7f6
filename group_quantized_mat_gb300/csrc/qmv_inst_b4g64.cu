// Kernels for bits = 4, group_size = 64.
#include "qmv_launch.cuh"

namespace qmv {
cudaError_t launch_b4g64_m1(const RingMaps &maps, const RingParams &p, const Launch &l, cudaStream_t stream)
{
    return launch_m1<4, 64>(maps, p, l, stream);
}
cudaError_t launch_b4g64_streamed(int V, const Params &p, const Launch &l, cudaStream_t stream)
{
    return launch_streamed<4, 64>(V, p, l, stream);
}
}  // namespace qmv
