// Launch table of the qmv kernels for one (bits, group_size) pair. Each
// qmv_inst_*.cu translation unit instantiates it once, so the four pairs
// compile in parallel.
#pragma once

#include <atomic>
#include <mutex>

#include "qmv_kernel.cuh"
#include "qmv_launch_decl.h"

namespace qmv {

static_assert(kConsumersV1 == kRingConsumers && kProducersV1 == kRingProducers, "launch bounds");
static_assert(kThreadsVN == kStreamedWarps * 32, "launch bounds");
static_assert(kOneWarps == kOneWarpsDecl && kOneCtasPerSm == kOneCtasPerSmDecl, "launch bounds");

template <typename Kern, typename... Args>
cudaError_t launch_one(Kern kern, std::atomic<int> (&configured)[64], const Launch &l, cudaStream_t stream, Args... args)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    // The opt-in dynamic shared-memory limit is a per-device kernel attribute;
    // raise it when this launch needs more than it was last set to. Raising
    // happens under a lock, so concurrent host threads never lower it under
    // each other; the cached value is stored only after the attribute is set.
    if (configured[dev].load() < int(l.smem)) {
        static std::mutex m;
        std::lock_guard<std::mutex> lock(m);
        if (configured[dev].load() < int(l.smem)) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(l.smem));
            if (e != cudaSuccess) return e;
            configured[dev].store(int(l.smem));
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = l.grid;
    cfg.blockDim = dim3(l.threads);
    cfg.dynamicSmemBytes = l.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = l.pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int BITS, int GS>
cudaError_t launch_m1(const RingMaps &maps, const RingParams &p, const Launch &l, cudaStream_t stream)
{
    static std::atomic<int> configured[2][64] = {};
    if (p.sb_packed) return launch_one(qmv_m1<BITS, GS, true>, configured[1], l, stream, maps.w, maps.s, maps.b, p);
    return launch_one(qmv_m1<BITS, GS, false>, configured[0], l, stream, maps.w, maps.s, maps.b, p);
}

template <int BITS, int GS, int V>
cudaError_t launch_ringv_v(const RingMaps &maps, const RingParams &p, const Launch &l, cudaStream_t stream)
{
    static std::atomic<int> configured[2][64] = {};
    if (p.sb_packed)
        return launch_one(qmv_ringv<BITS, GS, true, V>, configured[1], l, stream, maps.w, maps.s, maps.b, p);
    return launch_one(qmv_ringv<BITS, GS, false, V>, configured[0], l, stream, maps.w, maps.s, maps.b, p);
}

template <int BITS, int GS>
cudaError_t launch_ringv(int V, const RingMaps &maps, const RingParams &p, const Launch &l, cudaStream_t stream)
{
    if (V == 2) return launch_ringv_v<BITS, GS, 2>(maps, p, l, stream);
    if (V == 3) return launch_ringv_v<BITS, GS, 3>(maps, p, l, stream);
    if (V == 4) return launch_ringv_v<BITS, GS, 4>(maps, p, l, stream);
    return cudaErrorInvalidValue;
}

template <int BITS, int GS>
cudaError_t launch_one_vector(const Params &p, const Launch &l, cudaStream_t stream)
{
    static std::atomic<int> configured[2][64] = {};
    if (p.sb_packed) return launch_one(qmv_one<BITS, GS, true>, configured[1], l, stream, p);
    return launch_one(qmv_one<BITS, GS, false>, configured[0], l, stream, p);
}

template <int BITS, int GS, int V>
cudaError_t launch_v(const Params &p, const Launch &l, cudaStream_t stream)
{
    static std::atomic<int> configured[2][64] = {};
    if (p.sb_packed) return launch_one(qmv_streamed<BITS, GS, V, true>, configured[1], l, stream, p);
    return launch_one(qmv_streamed<BITS, GS, V, false>, configured[0], l, stream, p);
}

// The call's x staging for the streamed kernel (one thread per eight
// elements of a vector).
template <int BITS>
cudaError_t launch_stage(const uint16_t *x, int K, int S_row, int V, uint8_t *out, unsigned *counters, int ncounters,
                         bool pdl, cudaStream_t stream)
{
    static std::atomic<int> configured[64] = {};
    const long long threads = (long long)V * S_row * 8;
    Launch l;
    l.grid = dim3(unsigned((threads + kStageThreads - 1) / kStageThreads));
    l.threads = kStageThreads;
    l.smem = 0;
    l.pdl = pdl;
    return launch_one(qmv_stage_x<BITS>, configured, l, stream, x, K, S_row, V, out, counters, ncounters);
}

template <int BITS, int GS>
cudaError_t launch_streamed(int V, const Params &p, const Launch &l, cudaStream_t stream)
{
    switch (V) {
#define QMV_CASE(v) \
    case v: return launch_v<BITS, GS, v>(p, l, stream);
        QMV_CASE(2) QMV_CASE(3) QMV_CASE(4) QMV_CASE(5) QMV_CASE(6) QMV_CASE(7) QMV_CASE(8)
        QMV_CASE(9) QMV_CASE(10) QMV_CASE(11) QMV_CASE(12) QMV_CASE(13) QMV_CASE(14) QMV_CASE(15) QMV_CASE(16)
#undef QMV_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmv
