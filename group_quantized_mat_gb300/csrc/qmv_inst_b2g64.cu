// Kernels for bits = 2, group_size = 64.
#include "qmv_launch.cuh"

namespace qmv {
cudaError_t launch_b2g64_m1(const RingMaps &maps, const RingParams &p, const Launch &l, cudaStream_t stream)
{
    return launch_m1<2, 64>(maps, p, l, stream);
}
cudaError_t launch_b2g64_one(const Params &p, const Launch &l, cudaStream_t stream)
{
    return launch_one_vector<2, 64>(p, l, stream);
}
cudaError_t launch_b2g64_streamed(int V, const Params &p, const Launch &l, cudaStream_t stream)
{
    return launch_streamed<2, 64>(V, p, l, stream);
}
cudaError_t launch_b2g64_stage(const uint16_t *x, int K, int S_row, int V, uint8_t *out, unsigned *counters,
                             int ncounters, bool pdl, cudaStream_t stream)
{
    return launch_stage<2>(x, K, S_row, V, out, counters, ncounters, pdl, stream);
}
cudaError_t launch_b2g64_ringv(int V, const RingMaps &maps, const RingParams &p, const Launch &l, cudaStream_t stream)
{
    return launch_ringv<2, 64>(V, maps, p, l, stream);
}
}  // namespace qmv
