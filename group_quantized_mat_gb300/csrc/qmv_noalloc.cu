// qmv_run_noalloc: the mat-vec without any device allocation.
//
// Some callers cannot call cudaMalloc: engines whose device memory all
// belongs to their own pool allocator (a private cudaMalloc fragments it and
// can fail under memory pressure), and latency-bound decode loops (cudaMalloc
// may synchronize the whole device). qmv_run allocates its workspace on first
// use, and qmv_run_ex needs a workspace the caller allocated; this entry point
// needs neither. The scratch that K-split launches use lives in one
// fixed-size array of this file instead.
#include <cuda_runtime.h>

#include <mutex>

#include "qmv.h"
#include "qmv_launch_decl.h"

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
// A failure is recorded for qmv_last_cuda_error() and cleared from the
// runtime's error slot, so that no later launch reports it as its own.
qmv_status scratch_address(int dev, void **out)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_address[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return qmv::record_cuda_failure("cudaGetSymbolAddress(noalloc scratch)",
                                            e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        }
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
    // The host-side errors of qmv_run, reported first and in its order.
    qmv_status st = qmv::check_run_args(w_q, scales, biases, x, y, M, N, K, bits, group_size, nullptr, 0u);
    if (st != QMV_OK) return st;
    const size_t need = qmv_workspace_size(M, N, K, bits, group_size);
    if (need > QMV_NOALLOC_SCRATCH_BYTES) return QMV_ERR_WORKSPACE;

    // The first call on a device resolves the array's address whatever the
    // problem, so that after one call of any shape no later call has set-up
    // work left to do.
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return qmv::record_cuda_failure("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return qmv::record_cuda_failure("device index >= 64", cudaErrorInvalidDevice);
    void *scratch = nullptr;
    st = scratch_address(dev, &scratch);
    if (st != QMV_OK) return st;
    // The array keeps whatever the previous call left; a call needs nothing
    // of it (each launch clears its own K-split tickets). A problem that needs
    // no scratch is handed no workspace at all.
    if (need == 0) return qmv_run_ex(w_q, scales, biases, x, y, M, N, K, bits, group_size, nullptr, 0, 0u, stream);
    return qmv_run_ex(w_q, scales, biases, x, y, M, N, K, bits, group_size, scratch, QMV_NOALLOC_SCRATCH_BYTES, 0u,
                      stream);
}
