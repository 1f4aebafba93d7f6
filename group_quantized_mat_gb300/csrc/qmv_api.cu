// Host side of the C ABI declared in include/qmv.h: argument validation, the
// launch plan (fixed K-chunks, CTA shape), workspace handling, the weight
// tensor map, and dispatch to the kernels (M = 1 -> qmv_m1, M = 2..16 ->
// qmv_streamed with V = M).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "qmv.h"
#include "qmv_launch_decl.h"
#include "qmv_plan.h"

namespace {

// Device error word set by kernels whose bounded wait ran out.
__device__ unsigned g_qmv_device_error;

constexpr int kMaxDevices = 64;

struct DeviceState {
    void *workspace = nullptr;
    size_t workspace_bytes = 0;
    unsigned *err = nullptr;
    int sms = 0;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

// Last CUDA failure seen by this thread's calls into the library.
thread_local char g_last_error[160] = "no CUDA error recorded";

qmv_status cuda_fail(const char *what, cudaError_t e)
{
    snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return QMV_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

qmv_status check_shape(int M, int N, int K, int bits, int gs, bool check_m)
{
    if (bits != 2 && bits != 4) return QMV_ERR_BITS;
    if (gs != 64 && gs != 128) return QMV_ERR_GROUP;
    if (N < 1 || N > (1 << 30) || K < 1 || K % gs != 0 || K > (1 << 24)) return QMV_ERR_SHAPE;
    if (check_m && (M < 1 || M > QMV_MAX_M)) return QMV_ERR_M_RANGE;
    return QMV_OK;
}

struct Problem {
    int M, N, K, bits, gs, G;
    int ks;         // K-chunks per row (fixes the order; a function of K and gs only)
    int V;          // vectors per launch
    int RW;         // rows per row block (one warp's rows)
    int cps;        // chunks per CTA: ks (all of K) or 1
    int RB, H;      // row blocks (at most) and chunk phases per CTA
    int warps;      // warps per CTA
    int NB;         // row blocks of the matrix
    int balanced;   // persistent grid with an even share of row blocks per CTA
    int grid_x;     // CTAs along the rows
    int stages;     // weight stages in flight per warp
    int gsm;        // groups of x staged per CTA
    int tile_rows, ntiles;
    int smem;       // dynamic shared memory per CTA
};

// Largest dynamic shared memory a CTA may use (static shared memory and
// reserved bytes kept aside).
constexpr int kSmemBudget = 227 * 1024 - 256;
// CTA count below which row tiles are halved to spread the work (about two per SM).
constexpr int kMinCtas = 304;

#if defined(QMV_TUNING)
// Tuning builds only: fixed launch shapes for sweeps (0 = automatic).
struct TuneOverride { int whole_k = 0, RB = 0, H = 0, stages = 0, R = 0; };
TuneOverride g_tune;
#endif

int pow2_floor(int v)
{
    int p = 1;
    while (p * 2 <= v) p *= 2;
    return p;
}

void finish(Problem &pr)
{
    pr.tile_rows = pr.RB * pr.RW;
    pr.smem = qmv::smem_layout(pr.bits, pr.gs, pr.V, pr.RW, pr.warps, pr.stages, pr.gsm, pr.cps, pr.tile_rows).total;
}

// Launch shape of a call. `sms` is the device's SM count, or 0 when unknown
// (then no persistent grid is planned). Whether a workspace is needed never
// depends on `sms`, so qmv_workspace_size can be answered without a GPU.
Problem plan(int V, int N, int K, int bits, int gs, int sms)
{
    Problem pr;
    pr.M = V; pr.V = V; pr.N = N; pr.K = K; pr.bits = bits; pr.gs = gs;
    pr.G = K / gs;
    pr.ks = qmv::chunk_count(K, gs);
    pr.RW = 8;
    pr.balanced = 0;
    const int mw = qmv::max_warps(V);
    int want_whole = -1, want_rb = 0, want_h = 0, want_stages = 0;
#if defined(QMV_TUNING)
    if (g_tune.stages >= 2 && g_tune.stages <= 16 && (g_tune.stages & (g_tune.stages - 1)) == 0)
        want_stages = g_tune.stages;
    want_whole = g_tune.whole_k ? (g_tune.whole_k > 0 ? 1 : 0) : -1;
    if (g_tune.whole_k == 2) want_whole = 2;
    want_rb = g_tune.RB;
    want_h = g_tune.H;
    if (V == 1 && (g_tune.R == 2 || g_tune.R == 4)) pr.RW = 4 * g_tune.R;
#endif
    const int sb = qmv::stage_bytes(bits, gs, pr.RW);
    pr.stages = want_stages ? want_stages : pow2_floor(8192 / sb > 2 ? 8192 / sb : 2);
    pr.NB = (N + pr.RW - 1) / pr.RW;
    // All of K in one CTA (no workspace) when x of all of K fits in shared memory.
    const bool whole_ok =
        want_whole != 0 && pr.ks <= qmv::kMaxChunksPerCta &&
        qmv::smem_layout(bits, gs, V, pr.RW, 1, pr.stages, pr.G, pr.ks, pr.RW).total + 8 * 8192 <= kSmemBudget;
    if (whole_ok) {
        pr.cps = pr.ks;
        pr.gsm = pr.G;
        // Persistent grid: every SM gets an even share of the row blocks.
        if (sms > 0 && want_whole != 1 && pr.NB >= sms) {
            pr.balanced = 1;
            pr.grid_x = sms;
            pr.RB = (pr.NB + sms - 1) / sms;
            pr.H = want_h ? want_h : 1;
            if (!want_h)
                while (pr.H < pr.ks && pr.RB * (pr.H + 1) <= mw) ++pr.H;
            pr.warps = pr.RB * pr.H < mw ? pr.RB * pr.H : mw;
            finish(pr);
            while (pr.smem > kSmemBudget && pr.warps > 1) {
                --pr.warps;
                finish(pr);
            }
            if (pr.smem <= kSmemBudget && pr.H <= pr.cps) {
                pr.ntiles = pr.grid_x;
                return pr;
            }
            pr.balanced = 0;
        }
        pr.H = want_h ? want_h : (pr.ks < mw ? pr.ks : mw);
        pr.RB = want_rb ? want_rb : (8 / pr.H > 1 ? 8 / pr.H : 1);
        if (pr.RB * pr.H > mw) pr.RB = mw / pr.H > 0 ? mw / pr.H : 1;
        if (!want_rb)
            while (pr.RB > 1 && (pr.NB + pr.RB - 1) / pr.RB < kMinCtas) pr.RB /= 2;
        pr.warps = pr.RB * pr.H;
        finish(pr);
        if (pr.smem <= kSmemBudget && pr.H <= pr.cps && pr.warps <= mw) {
            pr.ntiles = pr.grid_x = (pr.NB + pr.RB - 1) / pr.RB;
            return pr;
        }
    }
    // Otherwise one chunk per CTA; chunk values meet in the workspace.
    pr.cps = 1;
    pr.H = 1;
    pr.gsm = qmv::chunk_groups(gs) < pr.G ? qmv::chunk_groups(gs) : pr.G;
    pr.RB = want_rb ? (want_rb < mw ? want_rb : mw) : (8 < mw ? 8 : mw);
    if (!want_rb)
        while (pr.RB > 1 && (pr.NB + pr.RB - 1) / pr.RB * pr.ks < kMinCtas) pr.RB /= 2;
    pr.warps = pr.RB;
    finish(pr);
    while (pr.smem > kSmemBudget && pr.stages > 2) {
        pr.stages /= 2;
        finish(pr);
    }
    pr.ntiles = pr.grid_x = (pr.NB + pr.RB - 1) / pr.RB;
    return pr;
}

size_t counter_bytes(int ntiles) { return (size_t(ntiles) * sizeof(unsigned) + 255) & ~size_t(255); }

size_t workspace_bytes_for(const Problem &pr)
{
    if (pr.cps == pr.ks) return 0;
    return counter_bytes(pr.ntiles) + size_t(pr.ks) * size_t(pr.V) * size_t(pr.N) * sizeof(float);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Weight matrix as a 2-D byte tensor [N rows, K*bits/8 bytes]; one box is
// 128 bytes x (rows per block), 128B-swizzled in shared memory.
int encode_weight_map(CUtensorMap *map, const uint32_t *w_q, const Problem &pr)
{
    auto fn = encode_fn();
    if (!fn) return -1;
    const cuuint64_t row_bytes = cuuint64_t(pr.K) * pr.bits / 8;
    const cuuint64_t dims[2] = {row_bytes, cuuint64_t(pr.N)};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {cuuint32_t(qmv::kBoxBytes), cuuint32_t(pr.RW)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t *>(w_q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return int(r);
}

qmv_status sm_count(int dev, int *out)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &d = g_devices[dev];
    if (!d.sms) {
        cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail("cudaDeviceGetAttribute(SM count)", e);
    }
    *out = d.sms;
    return QMV_OK;
}

qmv_status device_error_ptr(int dev, unsigned **out)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &d = g_devices[dev];
    if (!d.err) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_qmv_device_error);
        if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress", e);
        d.err = static_cast<unsigned *>(p);
    }
    *out = d.err;
    return QMV_OK;
}

// Library-owned workspace of `dev`, grown (and zero-filled) on demand.
qmv_status library_workspace(int dev, size_t need, void **out)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &d = g_devices[dev];
    if (d.workspace_bytes < need) {
        if (d.workspace) {
            cudaFree(d.workspace);
            d.workspace = nullptr;
            d.workspace_bytes = 0;
        }
        void *p = nullptr;
        cudaError_t e = cudaMalloc(&p, need);
        if (e != cudaSuccess) return cuda_fail("cudaMalloc(workspace)", e);
        e = cudaMemset(p, 0, need);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            cudaFree(p);
            return cuda_fail("cudaMemset(workspace)", e);
        }
        d.workspace = p;
        d.workspace_bytes = need;
    }
    *out = d.workspace;
    return QMV_OK;
}

cudaError_t dispatch(const Problem &pr, const CUtensorMap &map, const qmv::Params &p, cudaStream_t stream)
{
    const dim3 grid(pr.grid_x, pr.ks / pr.cps);
    const int threads = 32 * pr.warps;
    const size_t smem = size_t(pr.smem);
    const int R = pr.RW / 4;
    if (pr.bits == 4 && pr.gs == 64) return qmv::launch_b4g64(pr.V, R, map, p, grid, threads, smem, stream);
    if (pr.bits == 4 && pr.gs == 128) return qmv::launch_b4g128(pr.V, R, map, p, grid, threads, smem, stream);
    if (pr.bits == 2 && pr.gs == 64) return qmv::launch_b2g64(pr.V, R, map, p, grid, threads, smem, stream);
    return qmv::launch_b2g128(pr.V, R, map, p, grid, threads, smem, stream);
}

qmv_status run_impl(const uint32_t *w_q, const uint16_t *scales, const uint16_t *biases, const uint16_t *x, void *y,
                    int M, int N, int K, int bits, int gs, void *workspace, size_t workspace_bytes, unsigned flags,
                    cudaStream_t stream)
{
    if (!w_q || !scales || !biases || !x || !y) return QMV_ERR_NULL;
    qmv_status st = check_shape(M, N, K, bits, gs, true);
    if (st != QMV_OK) return st;
    if (flags & ~(QMV_F32_OUT | QMV_FORCE_M1_PER_COLUMN)) return QMV_ERR_FLAGS;
    const bool f32_out = (flags & QMV_F32_OUT) != 0;
    if (!aligned(w_q, 16) || !aligned(x, 16) || !aligned(scales, 2) || !aligned(biases, 2) ||
        !aligned(y, f32_out ? 4 : 2) || (workspace && !aligned(workspace, 16)))
        return QMV_ERR_ALIGN;

    const bool per_column = (flags & QMV_FORCE_M1_PER_COLUMN) != 0;
    const int V = per_column ? 1 : M;

    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail("cudaGetDevice", ce);
    if (dev >= kMaxDevices) return cuda_fail("device index >= 64", cudaErrorInvalidDevice);
    int sms = 0;
    st = sm_count(dev, &sms);
    if (st != QMV_OK) return st;
    const Problem pr = plan(V, N, K, bits, gs, sms);
    const size_t need = workspace_bytes_for(pr);
    if (need > 0) {
        if (workspace) {
            if (workspace_bytes < need) return QMV_ERR_WORKSPACE;
        } else {
            st = library_workspace(dev, need, &workspace);
            if (st != QMV_OK) return st;
        }
    }
    unsigned *err = nullptr;
    st = device_error_ptr(dev, &err);
    if (st != QMV_OK) return st;

    CUtensorMap map;
    const int enc = encode_weight_map(&map, w_q, pr);
    if (enc != 0) {
        snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled(weights) returned %d%s", enc,
                 enc < 0 ? " (driver entry point not found)" : "");
        return QMV_ERR_CUDA;
    }

    qmv::Params p;
    p.scales = scales;
    p.biases = biases;
    p.err = err;
    p.N = N; p.K = K; p.G = pr.G; p.ks = pr.ks; p.cps = pr.cps; p.RB = pr.RB; p.H = pr.H;
    p.warps = pr.warps; p.NB = pr.NB; p.balanced = pr.balanced;
    p.stages = pr.stages; p.gsm = pr.gsm; p.ntiles = pr.ntiles;
    p.f32_out = f32_out ? 1 : 0;
    p.counters = need ? static_cast<unsigned *>(workspace) : nullptr;
    p.partials = need ? reinterpret_cast<float *>(static_cast<char *>(workspace) + counter_bytes(pr.ntiles)) : nullptr;

    const size_t ysize = f32_out ? sizeof(float) : sizeof(uint16_t);
    const int launches = per_column ? M : 1;
    for (int m = 0; m < launches; ++m) {
        p.x = x + size_t(m) * K;
        p.y = static_cast<char *>(y) + size_t(m) * N * ysize;
        ce = dispatch(pr, map, p, stream);
        if (ce != cudaSuccess) return cuda_fail("kernel launch", ce);
    }
    return QMV_OK;
}

}  // namespace

extern "C" int qmv_split_count(int N, int K, int bits, int group_size)
{
    if (check_shape(1, N, K, bits, group_size, false) != QMV_OK) return 0;
    return qmv::chunk_count(K, group_size);
}

#if defined(QMV_TUNING)
extern "C" __attribute__((visibility("default"))) void qmv_tune_set(int whole_k, int RB, int H, int stages, int R)
{
    g_tune.whole_k = whole_k;
    g_tune.RB = RB;
    g_tune.H = H;
    g_tune.stages = stages;
    g_tune.R = R;
}
#endif

extern "C" size_t qmv_workspace_size(int M, int N, int K, int bits, int group_size)
{
    if (check_shape(M, N, K, bits, group_size, true) != QMV_OK) return 0;
    return workspace_bytes_for(plan(M, N, K, bits, group_size, 0));
}

extern "C" qmv_status qmv_run(const uint32_t *w_q, const uint16_t *scales, const uint16_t *biases, const uint16_t *x,
                              uint16_t *y, int M, int N, int K, int bits, int group_size, qmv_stream_t stream)
{
    return run_impl(w_q, scales, biases, x, y, M, N, K, bits, group_size, nullptr, 0, 0u,
                    reinterpret_cast<cudaStream_t>(stream));
}

extern "C" qmv_status qmv_run_ex(const uint32_t *w_q, const uint16_t *scales, const uint16_t *biases,
                                 const uint16_t *x, void *y, int M, int N, int K, int bits, int group_size,
                                 void *workspace, size_t workspace_bytes, unsigned flags, qmv_stream_t stream)
{
    return run_impl(w_q, scales, biases, x, y, M, N, K, bits, group_size, workspace, workspace_bytes, flags,
                    reinterpret_cast<cudaStream_t>(stream));
}

extern "C" qmv_status qmv_workspace_init(void *workspace, size_t bytes, qmv_stream_t stream)
{
    if (!workspace) return bytes == 0 ? QMV_OK : QMV_ERR_NULL;
    if (!aligned(workspace, 16)) return QMV_ERR_ALIGN;
    cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QMV_OK : cuda_fail("cudaMemsetAsync(workspace)", e);
}

extern "C" qmv_status qmv_device_error(unsigned *word)
{
    if (!word) return QMV_ERR_NULL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail("cudaDeviceSynchronize", e);
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_qmv_device_error, sizeof v);
    if (e != cudaSuccess) return cuda_fail("cudaMemcpyFromSymbol", e);
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_qmv_device_error, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail("cudaMemcpyToSymbol", e);
    *word = v;
    return QMV_OK;
}

extern "C" const char *qmv_last_cuda_error(void) { return g_last_error; }

extern "C" const char *qmv_status_string(qmv_status s)
{
    switch (s) {
        case QMV_OK: return "QMV_OK";
        case QMV_ERR_NULL: return "QMV_ERR_NULL: a required pointer is NULL";
        case QMV_ERR_BITS: return "QMV_ERR_BITS: bits must be 2 or 4";
        case QMV_ERR_GROUP: return "QMV_ERR_GROUP: group_size must be 64 or 128";
        case QMV_ERR_SHAPE: return "QMV_ERR_SHAPE: need 1 <= N <= 2^30, 1 <= K <= 2^24, K % group_size == 0";
        case QMV_ERR_M_RANGE: return "QMV_ERR_M_RANGE: M must be in [1, 16]";
        case QMV_ERR_ALIGN: return "QMV_ERR_ALIGN: w_q, x and workspace need 16-byte alignment, scales/biases/y 2 (f32 y: 4)";
        case QMV_ERR_CUDA: return "QMV_ERR_CUDA: a CUDA runtime call or kernel launch failed";
        case QMV_ERR_WORKSPACE: return "QMV_ERR_WORKSPACE: workspace smaller than qmv_workspace_size()";
        case QMV_ERR_VALUE: return "QMV_ERR_VALUE: a quantized value does not fit in `bits` bits";
        case QMV_ERR_FLAGS: return "QMV_ERR_FLAGS: unknown flag bits";
    }
    return "unknown qmv_status";
}
