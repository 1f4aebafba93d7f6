// Entry points of the per-(bits, group_size) kernel tables (qmv_inst_*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "qmv.h"
#include "qmv_plan.h"

namespace qmv {

// Warps per CTA of the streamed kernel (its launch bounds), and the one-vector
// kernel's consumer and producer warps.
constexpr int kStreamedWarps = 12;
constexpr int kRingConsumers = 16;
constexpr int kRingProducers = 4;
// The one-vector kernel qmv_one: warps per CTA and CTAs per SM.
constexpr int kOneWarpsDecl = 12;
constexpr int kOneCtasPerSmDecl = 1;

// Tensor maps of the one-vector kernel: weights (tiles only), scales, biases.
struct RingMaps {
    CUtensorMap w, s, b;
};

struct Launch {
    dim3 grid;
    int threads;
    size_t smem;
    bool pdl;  // launch with a programmatic dependency on the preceding grid
};

// Arguments of the mxfp4 kernel (E2M1 codes, one E8M0 byte per 32 along K).
struct MxParams {
    const uint32_t *w;       // codes [N][K / 8] words, 8 per word, element 0 in the low nibble
    const uint8_t *scales;   // E8M0 bytes [N][K / 32]
    const uint16_t *x;       // bf16 [V][K]
    void *y;                 // bf16 (or fp32 with f32_out) [V][N]
    int N, K;                // K a multiple of 32
    int f32_out;
};

// Host-side argument checks of qmv_run_ex (QMV_OK or the status it would
// return, nothing launched), and recording a CUDA failure as the calling
// thread's qmv_last_cuda_error() text (returns QMV_ERR_CUDA). qmv_api.cu.
qmv_status check_run_args(const void *w_q, const void *scales, const void *biases, const void *x, const void *y,
                          int M, int N, int K, int bits, int gs, const void *workspace, unsigned flags);
qmv_status record_cuda_failure(const char *what, cudaError_t e);

// One launch for V = 1..16 vectors (qmv_mx.cu).
cudaError_t launch_mxfp4(int V, const MxParams &p, cudaStream_t stream);

#define QMV_DECLARE_LAUNCH(name)                                                                                  \
    cudaError_t name##_m1(const RingMaps &maps, const RingParams &p, const Launch &l, cudaStream_t stream);      \
    cudaError_t name##_one(const Params &p, const Launch &l, cudaStream_t stream);                               \
    cudaError_t name##_ringv(int V, const RingMaps &maps, const RingParams &p, const Launch &l, cudaStream_t stream); \
    cudaError_t name##_streamed(int V, const Params &p, const Launch &l, cudaStream_t stream);                   \
    cudaError_t name##_stage(const uint16_t *x, int K, int S_row, int V, uint8_t *out, unsigned *counters,       \
                             int ncounters, bool pdl, cudaStream_t stream);
QMV_DECLARE_LAUNCH(launch_b4g64)
QMV_DECLARE_LAUNCH(launch_b4g128)
QMV_DECLARE_LAUNCH(launch_b2g64)
QMV_DECLARE_LAUNCH(launch_b2g128)
#undef QMV_DECLARE_LAUNCH

}  // namespace qmv
