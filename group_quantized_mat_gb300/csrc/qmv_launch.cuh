// Launch table of the qmv kernels for one (bits, group_size) pair. Each
// qmv_inst_*.cu translation unit instantiates it once, so the four pairs
// compile in parallel.
#pragma once

#include "qmv_kernel.cuh"
#include "qmv_launch_decl.h"

namespace qmv {

template <typename Kern>
cudaError_t launch_one(Kern kern, int (&configured)[64], const CUtensorMap &map, const Params &p, dim3 grid,
                       int threads, size_t smem, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    // The opt-in dynamic shared-memory limit is a per-device kernel attribute;
    // raise it when this launch needs more than it was last set to.
    if (configured[dev] < int(smem)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = int(smem);
    }
    kern<<<grid, threads, smem, stream>>>(map, p);
    return cudaGetLastError();
}

template <int BITS, int GS, int V>
cudaError_t launch_v(int R, const CUtensorMap &map, const Params &p, dim3 grid, int threads, size_t smem,
                     cudaStream_t stream)
{
    if constexpr (V == 1) {
        static int configured2[64] = {0}, configured4[64] = {0};
        if (R == 4) return launch_one(qmv_m1<BITS, GS, 4>, configured4, map, p, grid, threads, smem, stream);
        return launch_one(qmv_m1<BITS, GS, 2>, configured2, map, p, grid, threads, smem, stream);
    } else {
        static int configured[64] = {0};
        return launch_one(qmv_streamed<BITS, GS, V>, configured, map, p, grid, threads, smem, stream);
    }
}

template <int BITS, int GS>
cudaError_t launch_bits_gs(int V, int R, const CUtensorMap &map, const Params &p, dim3 grid, int threads,
                           size_t smem, cudaStream_t stream)
{
    switch (V) {
#define QMV_CASE(v) \
    case v: return launch_v<BITS, GS, v>(R, map, p, grid, threads, smem, stream);
        QMV_CASE(1) QMV_CASE(2) QMV_CASE(3) QMV_CASE(4) QMV_CASE(5) QMV_CASE(6) QMV_CASE(7) QMV_CASE(8)
        QMV_CASE(9) QMV_CASE(10) QMV_CASE(11) QMV_CASE(12) QMV_CASE(13) QMV_CASE(14) QMV_CASE(15) QMV_CASE(16)
#undef QMV_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmv
