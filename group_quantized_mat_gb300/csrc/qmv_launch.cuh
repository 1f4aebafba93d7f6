// Launch table of the qmv kernels for one (bits, group_size) pair. Each
// qmv_inst_*.cu translation unit instantiates it once, so the four pairs
// compile in parallel.
#pragma once

#include "qmv_kernel.cuh"
#include "qmv_launch_decl.h"

namespace qmv {

// Per device and kernel: the dynamic shared memory the kernel is configured
// for, and the resident CTAs per SM at that size.
struct KernelCache {
    int smem[64] = {0};
    int per_sm[64] = {0};
};

template <typename Kern>
cudaError_t launch_one(Kern kern, KernelCache &cache, const CUtensorMap &map, Params p, int grid_y, size_t smem,
                       cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    if (cache.smem[dev] != int(smem)) {
        // The opt-in dynamic shared-memory limit is a per-device kernel attribute.
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
        if (e != cudaSuccess) return e;
        cache.per_sm[dev] = per_sm > 0 ? per_sm : 1;
        cache.smem[dev] = int(smem);
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // Persistent CTAs: as many as are resident at once, each looping over row tiles.
    int gx = cache.per_sm[dev] * sms / grid_y;
    if (gx < 1) gx = 1;
    if (gx > p.ntiles) gx = p.ntiles;
    kern<<<dim3(gx, grid_y), kThreads, smem, stream>>>(map, p);
    return cudaGetLastError();
}

template <int BITS, int GS, int V>
cudaError_t launch_v(const CUtensorMap &map, const Params &p, int grid_y, size_t smem, cudaStream_t stream)
{
    static KernelCache cache;
    if constexpr (V == 1)
        return launch_one(qmv_m1<BITS, GS>, cache, map, p, grid_y, smem, stream);
    else
        return launch_one(qmv_streamed<BITS, GS, V>, cache, map, p, grid_y, smem, stream);
}

template <int BITS, int GS>
cudaError_t launch_bits_gs(int V, const CUtensorMap &map, const Params &p, int grid_y, size_t smem,
                           cudaStream_t stream)
{
    switch (V) {
#define QMV_CASE(v) \
    case v: return launch_v<BITS, GS, v>(map, p, grid_y, smem, stream);
        QMV_CASE(1) QMV_CASE(2) QMV_CASE(3) QMV_CASE(4) QMV_CASE(5) QMV_CASE(6) QMV_CASE(7) QMV_CASE(8)
        QMV_CASE(9) QMV_CASE(10) QMV_CASE(11) QMV_CASE(12) QMV_CASE(13) QMV_CASE(14) QMV_CASE(15) QMV_CASE(16)
#undef QMV_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmv
