// qmv_run_noalloc: the mat-vec without any device allocation.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured (an allocation there is not stream-ordered and breaks or
// serializes the capture), engines whose device memory all belongs to their
// own pool allocator (a private cudaMalloc fragments it and can fail under
// memory pressure), and latency-bound decode loops (cudaMalloc may
// synchronize the whole device). qmv_run allocates its workspace on first
// use, and qmv_run_ex needs a workspace the caller allocated; this entry point
// needs neither. The scratch that K-split launches use lives in one
// fixed-size array of this file instead.
#include <cuda_runtime.h>

#include <mutex>

#include "qmv.h"

namespace {

// Scratch shared by every qmv_run_noalloc call on a device. Each GPU that
// loads this library holds QMV_NOALLOC_SCRATCH_BYTES of it until the process
// exits. It keeps whatever the last call left in it, which no call reads.
__device__ __align__(256) unsigned char g_noalloc_scratch[QMV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_address[kMaxDevices] = {nullptr};

// In host code the array's name is only a host-side stand-in, never a device
// address: resolve the real address once per device, with that device current.
qmv_status scratch_address(int dev, void **out)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_address[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return QMV_ERR_CUDA;
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return QMV_OK;
}

}  // namespace

extern "C" qmv_status qmv_run_noalloc(const uint32_t *w_q, const uint16_t *scales, const uint16_t *biases,
                                      const uint16_t *x, uint16_t *y, int M, int N, int K, int bits,
                                      int group_size, qmv_stream_t stream)
{
    const size_t need = qmv_workspace_size(M, N, K, bits, group_size);
    if (need > QMV_NOALLOC_SCRATCH_BYTES) return QMV_ERR_WORKSPACE;
    // No scratch needed (or invalid arguments, which qmv_run_ex rejects on the
    // host before it could touch any workspace): nothing to set up.
    if (need == 0) return qmv_run_ex(w_q, scales, biases, x, y, M, N, K, bits, group_size, nullptr, 0, 0u, stream);

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMV_ERR_CUDA;
    void *scratch = nullptr;
    qmv_status st = scratch_address(dev, &scratch);
    if (st != QMV_OK) return st;
    // The array keeps whatever the previous call left; a call needs nothing
    // of it (each launch clears its own K-split tickets).
    return qmv_run_ex(w_q, scales, biases, x, y, M, N, K, bits, group_size, scratch, QMV_NOALLOC_SCRATCH_BYTES, 0u,
                      stream);
}
