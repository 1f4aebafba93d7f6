// Host side of the C ABI declared in include/qmv.h: argument validation, the
// launch plans (fixed K-chunks, CTA shape, the one-vector kernel's ring),
// workspace handling, the scale/bias tensor maps and dispatch to the kernels
// (M = 1 -> qmv_m1, M = 2..16 -> qmv_streamed with V = M), and the mxfp4
// entry point (qmv_mxfp4 in qmv_mx.cu for every M).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
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
    // scale / bias element indices and weight byte offsets stay within 31 and 47 bits
    if ((long long)N * (K / gs) >= (1ll << 31)) return QMV_ERR_SHAPE;
    if (check_m && (M < 1 || M > QMV_MAX_M)) return QMV_ERR_M_RANGE;
    return QMV_OK;
}

struct Problem {
    int V, N, K, bits, gs, G;
    int S_row;      // 64-element subgroups per row
    int ks;         // K-chunks per row (fixes the order; a function of K only)
    int row_bytes;
    int NB;         // row blocks of 4 rows
    int cpc;        // chunks per CTA
    int nranges;    // chunk ranges (grid.y)
    int grid_rows;  // CTAs along the rows (grid.x)
    int max_rb;     // row blocks of the largest CTA share
    int threads;
    int smem;       // dynamic shared memory per CTA
    // one-vector ring
    int uc, unit_mode, pitch, sb_mode_unit, sbox, slots, consumers;
    int ringv;      // 2..4 vectors through the ring (staged cells from the workspace)
    int sb_packed;
};

// Largest dynamic shared memory a CTA may use (static shared memory and
// reserved bytes kept aside).
constexpr int kSmemBudget = 227 * 1024 - 512;
// Chunk values of one CTA at most (bounds its share of rows).
constexpr int kCvBudget = 16 * 1024;
// One-vector kernel: staged x at most, largest unit, ring depth.
constexpr int kXsBudgetV1 = 80 * 1024;
constexpr int kUnitMax = 8 * 1024;
// Whole-row units may be up to 10 KB (four rows of K = 5120 at 4 bits) when
// every consumer warp gets at least two of them: a 17408 x 5120 matrix then
// runs 3 % faster on the ring than on the direct-load kernel, while 5120 x 5120
// (one unit per consumer) runs 15 % slower.
constexpr int kUnitMaxRows = 10 * 1024;
constexpr int kMaxSlots = 32;
// Rows at least this long go to the ring whatever their unit shape.
constexpr int kRingMinK = 12288;


// The widest chunk range that fits (cpc_max) split into equal ranges: as many
// ranges as cpc_max needs, each ceil(ks / ranges) chunks, so that no CTA
// carries a much longer range than another.
int balanced_cpc(int ks, int cpc_max)
{
    if (cpc_max < 1) cpc_max = 1;
    const int nranges = (ks + cpc_max - 1) / cpc_max;
    return (ks + nranges - 1) / nranges;
}

void common_shape(Problem &pr, int V, int N, int K, int bits, int gs)
{
    pr.V = V; pr.N = N; pr.K = K; pr.bits = bits; pr.gs = gs;
    pr.G = K / gs;
    pr.S_row = qmv::subs_per_row(K);
    pr.ks = qmv::chunk_count(K);
    pr.row_bytes = int((long long)K * bits / 8);
    pr.NB = (N + qmv::kRows - 1) / qmv::kRows;
}

// A persistent grid of about one CTA per SM: the chunk ranges times an even
// split of the row blocks; more CTAs (several waves) when a share of rows
// would exceed what `cv_bytes` of chunk values hold.
void grid_shape(Problem &pr, int sms, int V, int cv_bytes)
{
    pr.nranges = (pr.ks + pr.cpc - 1) / pr.cpc;
    int gr = sms > 0 ? sms / pr.nranges : 1;
    if (gr < 1) gr = 1;
    const int per_rb = qmv::kRows * pr.cpc * V * 4;
    const int rb_cap = cv_bytes / per_rb > 0 ? cv_bytes / per_rb : 1;
    if ((pr.NB + gr - 1) / gr > rb_cap) gr = (pr.NB + rb_cap - 1) / rb_cap;
    if (gr > pr.NB) gr = pr.NB;
    pr.grid_rows = gr;
    pr.max_rb = (pr.NB + gr - 1) / gr;
}

// Streamed kernel (V >= 2): all of K per CTA (no K split) when the x cells
// of all of K fit, else the widest chunk range that fits (one chunk always
// does). Whether the K split happens never depends on `sms` (the fit is
// checked against the chunk-value cap), so qmv_workspace_size needs no GPU.
Problem plan_direct(int V, int N, int K, int bits, int gs, int sms)
{
    Problem pr{};
    common_shape(pr, V, N, K, bits, gs);
    auto nsub_of = [&](int cpc) { return cpc * qmv::kChunkSubs < pr.S_row ? cpc * qmv::kChunkSubs : pr.S_row; };
    auto xs_bytes = [&](int cpc) { return qmv::align_up(V * nsub_of(cpc) * qmv::kXsF32, 16); };
    // Two or three vectors whose cells of all of K fit half the shared memory:
    // CTAs of 8 warps, two per SM (their registers allow it), so more warps
    // cover each other's weight loads (15360 x 3840 at M = 2: 17.3 -> 15.8 us).
    // Where that would split K (3840 x 15360), the split cost more than the
    // warps gained.
    const int half = kSmemBudget / 2 - 256;
    const int per_sm = V <= 3 && xs_bytes(pr.ks) + kCvBudget + 16 + 128 <= half ? 2 : 1;
    const int warps = per_sm == 2 ? 8 : qmv::kStreamedWarps;
    const int budget = per_sm == 2 ? half : kSmemBudget;
    const int wbuf = qmv::vectors_per_pass(V) < V ? warps * qmv::kRows * 32 * qmv::sub_bytes(bits) : 0;
    pr.cpc = pr.ks;
    while (pr.cpc > 1 && xs_bytes(pr.cpc) + kCvBudget + wbuf + 16 + 128 > budget) --pr.cpc;
    pr.cpc = balanced_cpc(pr.ks, pr.cpc);
    pr.threads = 32 * warps;
    // chunk values may use whatever shared memory the x cells and the weight
    // buffer leave (at least kCvBudget, by the fit above)
    grid_shape(pr, per_sm * sms, V, budget - (xs_bytes(pr.cpc) + wbuf + 16 + 128 + 16));
    pr.smem = qmv::smem_layout(bits, V, warps, nsub_of(pr.cpc), pr.max_rb, pr.cpc).total;
    return pr;
}

// One-vector kernel: chunks per CTA from the staged-x budget (all of K when
// it fits), units (whole rows in one copy when four rows fit kUnitMax, else
// uc chunks of each row: one 2-D box of the 4 rows when the scale/bias rows
// are 16-byte multiples, else one copy per row), scale/bias boxes, then as
// many ring slots as fit (a multiple of the producer warps, at most kMaxSlots
// and the CTA's units).
Problem plan_ring(int N, int K, int bits, int gs, int sms, bool sb_packed, int V = 1)
{
    Problem pr{};
    common_shape(pr, V, N, K, bits, gs);
    // raw x (128 bytes a subgroup) and its staged cell (kXsB16 bytes); V >= 2:
    // the V staged fp32 cells
    const int per_sub = V == 1 ? 128 + qmv::kXsB16 : V * qmv::kXsF32;
    pr.cpc = pr.S_row * per_sub <= kXsBudgetV1 ? pr.ks : balanced_cpc(pr.ks, kXsBudgetV1 / (qmv::kChunkSubs * per_sub));
    pr.consumers = qmv::kRingConsumers;
    grid_shape(pr, sms, V, kCvBudget);
    const int cb = qmv::chunk_bytes(bits);
    bool whole = pr.cpc == pr.ks && qmv::kRows * pr.row_bytes <= kUnitMaxRows;
    if (whole) {
        pr.unit_mode = qmv::kUnitRows;
        pr.uc = pr.ks;
        pr.pitch = pr.row_bytes;
    } else {
        // a tile row is at most 256 eight-byte elements (kUnitMax / 4 rows)
        pr.unit_mode = pr.G * qmv::sb_elem_bytes(sb_packed) % 16 == 0 ? qmv::kUnitTiles : qmv::kUnitPieces;
        pr.uc = kUnitMax / (qmv::kRows * cb);
        if (pr.uc < 1) pr.uc = 1;
        if (pr.uc > pr.cpc) pr.uc = pr.cpc;
        pr.pitch = pr.uc * cb;
    }
    // Scale/bias boxes: one per unit when the four rows' groups fit one box,
    // else one per row. A box starts at a multiple of 8 elements, so it spans
    // up to 7 more.
    const int gpu = pr.unit_mode == qmv::kUnitRows
                        ? pr.G
                        : (pr.uc * qmv::kChunkElems / gs < pr.G ? pr.uc * qmv::kChunkElems / gs : pr.G);
    pr.sb_packed = sb_packed ? 1 : 0;
    const int A = 16 / qmv::sb_elem_bytes(pr.sb_packed);  // box start alignment, elements
    if (pr.unit_mode == qmv::kUnitTiles) {
        pr.sb_mode_unit = 1;
        pr.sbox = qmv::kRows * (pr.uc * qmv::kChunkElems / gs);  // 4 box rows, each the unit's groups
    } else if (pr.unit_mode == qmv::kUnitRows && qmv::kRows * pr.G + A - 1 <= 256) {
        pr.sb_mode_unit = 1;
        pr.sbox = qmv::align_up(qmv::kRows * pr.G + A - 1, A);
    } else {
        pr.sb_mode_unit = 0;
        pr.sbox = qmv::align_up(gpu + A - 1, A);
    }
    const int nsub = pr.cpc * qmv::kChunkSubs < pr.S_row ? pr.cpc * qmv::kChunkSubs : pr.S_row;
    auto layout = [&](int slots) {
        return qmv::ring_layout(pr.pitch, pr.sb_mode_unit, pr.sbox, pr.sb_packed, slots, nsub, pr.max_rb, pr.cpc, V);
    };
    // Slots: a multiple of the producer and the consumer counts (each slot
    // has one producer and one consumer warp). A consumer warp with a single
    // slot waits a full memory latency between its units, so the largest
    // consumer count whose ring gives every consumer two slots is taken;
    // failing that, one slot per consumer (fewer consumers if even that does
    // not fit).
    const int P = qmv::kRingProducers;
    int C = 0;
    const int cmax = V == 1 ? qmv::kRingConsumers : 12;
    for (int c : {qmv::kRingConsumers, 12, 8})
        if (c <= cmax && layout(2 * c).total <= kSmemBudget) {
            C = c;
            break;
        }
    if (C == 0) {
        C = cmax;
        while (C > P && layout(C).total > kSmemBudget) C /= 2;
    }
    int slots = C;
    while (slots + C <= kMaxSlots && layout(slots + C).total <= kSmemBudget) slots += C;
    pr.consumers = C;
    pr.slots = slots;
    pr.smem = layout(slots).total;
    pr.threads = 32 * (C + P);
    return pr;
}

// One-vector kernel qmv_one: all of K per CTA when its staged x fits the
// budget, else the widest chunk range that does; about kOneCtasPerSm CTAs per
// SM. Like plan_direct, the K split never depends on `sms`.
constexpr int kUnitOne = -1;  // unit_mode of a qmv_one plan
constexpr int kXsBudgetOne = 48 * 1024;
constexpr int kCvBudgetOne = 8 * 1024;

Problem plan_one(int N, int K, int bits, int gs, int sms, bool sb_packed)
{
    Problem pr{};
    common_shape(pr, 1, N, K, bits, gs);
    const int per_chunk = qmv::kChunkSubs * qmv::kXsB16;
    pr.cpc = pr.S_row * qmv::kXsB16 <= kXsBudgetOne ? pr.ks : balanced_cpc(pr.ks, kXsBudgetOne / per_chunk);
    grid_shape(pr, sms * qmv::kOneCtasPerSmDecl, 1, kCvBudgetOne);
    pr.threads = 32 * qmv::kOneWarpsDecl;
    const int nsub = pr.cpc * qmv::kChunkSubs < pr.S_row ? pr.cpc * qmv::kChunkSubs : pr.S_row;
    pr.smem = qmv::one_layout(nsub, pr.max_rb, pr.cpc).total;
    pr.unit_mode = kUnitOne;
    pr.sb_packed = sb_packed ? 1 : 0;
    return pr;
}

Problem plan(int V, int N, int K, int bits, int gs, int sms, bool sb_packed = false)
{
    if (V >= 2) {
        // 2..4 vectors over whole-row units: the ring, consumers running the
        // packed-fma datapath on the call's staged cells
        if (V <= 4 && (long long)qmv::kRows * K * bits / 8 <= kUnitMax) {
            Problem pr = plan_ring(N, K, bits, gs, sms, sb_packed, V);
            if (pr.unit_mode == qmv::kUnitRows && pr.cpc == pr.ks && pr.consumers >= 4) {
                pr.ringv = 1;
                return pr;
            }
        }
        return plan_direct(V, N, K, bits, gs, sms);
    }
    // One vector: the ring when a unit is four whole rows in one copy, or
    // for long rows (where staging x once per SM, not per CTA, matters);
    // otherwise the direct-load kernel, whose units need no per-row copies.
    const long long four_rows = (long long)qmv::kRows * K * bits / 8;
    if (four_rows <= kUnitMax || K >= kRingMinK) return plan_ring(N, K, bits, gs, sms, sb_packed);
    if (four_rows <= kUnitMaxRows) {
        // whole-row units of up to 10 KB, if each consumer warp gets two
        const Problem pr = plan_ring(N, K, bits, gs, sms, sb_packed);
        if (pr.unit_mode == qmv::kUnitRows && (long long)pr.NB >= 2LL * pr.consumers * pr.grid_rows) return pr;
    }
    return plan_one(N, K, bits, gs, sms, sb_packed);
}

size_t counter_bytes(int NB) { return (size_t(NB) * sizeof(unsigned) + 255) & ~size_t(255); }

// Workspace of a launch: [counters][partials] when CTAs split K, then for the
// streamed kernel the call's staged x cells [V][S_row]. Nothing in it carries
// over between calls: each launch clears its tickets first.
size_t split_bytes(const Problem &pr)
{
    if (pr.cpc >= pr.ks) return 0;
    return counter_bytes(pr.NB) + size_t(pr.ks) * size_t(pr.V) * size_t(pr.N) * sizeof(float);
}
size_t align256(size_t b) { return (b + 255) & ~size_t(255); }
size_t staged_offset(const Problem &pr) { return align256(split_bytes(pr)); }
size_t workspace_bytes_for(const Problem &pr)
{
    if (pr.V < 2) return split_bytes(pr);
    return staged_offset(pr) + align256(size_t(pr.V) * size_t(pr.S_row) * size_t(qmv::kXsF32));
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

// Scales or biases (or the interleaved pairs, 4-byte elements): for tiles a
// 2-D tensor [N][G] whose box is 4 rows of sbox / 4 groups, else a 1-D tensor
// of N*G elements whose box is `sbox` elements. Elements outside the tensor
// arrive as zeros.
int encode_sb_map(CUtensorMap *map, const uint16_t *base, const Problem &pr)
{
    auto fn = encode_fn();
    if (!fn) return -1;
    CUresult r;
    const auto dtype = pr.sb_packed ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
    if (pr.unit_mode == qmv::kUnitTiles) {
        const cuuint64_t dims[2] = {cuuint64_t(pr.G), cuuint64_t(pr.N)};
        // a multiple of 16 bytes (the planner's condition for tiles)
        const cuuint64_t strides[1] = {cuuint64_t(pr.G) * cuuint64_t(qmv::sb_elem_bytes(pr.sb_packed))};
        const cuuint32_t box[2] = {cuuint32_t(pr.sbox / qmv::kRows), cuuint32_t(qmv::kRows)};
        const cuuint32_t estr[2] = {1, 1};
        r = fn(map, dtype, 2, const_cast<uint16_t *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[1] = {cuuint64_t(pr.N) * cuuint64_t(pr.G)};
        const cuuint64_t strides[1] = {0};
        const cuuint32_t box[1] = {cuuint32_t(pr.sbox)};
        const cuuint32_t estr[1] = {1};
        r = fn(map, dtype, 1, const_cast<uint16_t *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return int(r);
}

// Packed weights as a 2-D tensor [N][row_bytes / 8] of 8-byte elements (a
// row is a multiple of 16 bytes); a box is 4 rows of `pitch` bytes. Bytes
// past a row's end and rows past N arrive as zeros.
int encode_w_map(CUtensorMap *map, const uint32_t *w_q, const Problem &pr)
{
    auto fn = encode_fn();
    if (!fn) return -1;
    const cuuint64_t dims[2] = {cuuint64_t(pr.row_bytes / 8), cuuint64_t(pr.N)};
    const cuuint64_t strides[1] = {cuuint64_t(pr.row_bytes)};
    const cuuint32_t box[2] = {cuuint32_t(pr.pitch / 8), cuuint32_t(qmv::kRows)};
    const cuuint32_t estr[2] = {1, 1};
    return int(fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint32_t *>(w_q), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
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

// Library-owned workspace of `dev`, grown on demand. It is scratch (every
// launch clears the tickets it uses on its own stream), so a new allocation
// needs no initialization. Growing frees the smaller one first: cudaFree
// waits for the device's work in flight, which may still be using it.
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
        d.workspace = p;
        d.workspace_bytes = need;
    }
    *out = d.workspace;
    return QMV_OK;
}

cudaError_t dispatch(const Problem &pr, const qmv::RingMaps &maps, const qmv::Params &p, bool pdl, cudaStream_t stream)
{
    qmv::Launch l;
    l.grid = dim3(pr.grid_rows, pr.nranges);
    l.threads = pr.threads;
    l.smem = size_t(pr.smem);
    l.pdl = pdl;
    if (pr.V >= 2) {
        // the call's x staging first; the streamed kernel follows it with a
        // programmatic dependency, so its weight loads overlap the staging
        // (everything it writes, and the staged cells it reads, come after
        // its wait for the staging grid, itself ordered after the stream's
        // earlier work)
        // (it also clears the K-split tickets)
        uint8_t *cells = const_cast<uint8_t *>(p.xs_staged);
        const int nc = p.counters ? pr.NB : 0;
        cudaError_t e;
        if (pr.bits == 4 && pr.gs == 64)
            e = qmv::launch_b4g64_stage(p.x, pr.K, pr.S_row, pr.V, cells, p.counters, nc, pdl, stream);
        else if (pr.bits == 4)
            e = qmv::launch_b4g128_stage(p.x, pr.K, pr.S_row, pr.V, cells, p.counters, nc, pdl, stream);
        else if (pr.gs == 64)
            e = qmv::launch_b2g64_stage(p.x, pr.K, pr.S_row, pr.V, cells, p.counters, nc, pdl, stream);
        else
            e = qmv::launch_b2g128_stage(p.x, pr.K, pr.S_row, pr.V, cells, p.counters, nc, pdl, stream);
        if (e != cudaSuccess) return e;
        l.pdl = true;
    } else if (p.counters) {
        // a K-split one-vector launch: its tickets start at zero
        cudaError_t e = cudaMemsetAsync(p.counters, 0, counter_bytes(pr.NB), stream);
        if (e != cudaSuccess) return e;
    }
    if (pr.V == 1 && !p.counters) {
        // A one-vector launch always carries a programmatic dependency: its
        // set-up (barriers, tensor maps, shared memory) overlaps the tail of
        // the preceding kernel, and it reads nothing before waiting for that
        // kernel unless QMV_PDL allows the weights to stream under it.
        l.pdl = true;
    }
    if (pr.ringv) {
        qmv::RingParams rp;
        static_cast<qmv::Params &>(rp) = p;
        rp.uc = pr.uc; rp.unit_mode = pr.unit_mode; rp.pitch = pr.pitch; rp.sb_mode_unit = pr.sb_mode_unit;
        rp.sbox = pr.sbox; rp.slots = pr.slots; rp.consumers = pr.consumers;
        // the staging kernel before it writes no weights and started after the
        // stream's earlier work completed: the weights may stream under it
        rp.early_weights = 1;
        if (pr.bits == 4 && pr.gs == 64) return qmv::launch_b4g64_ringv(pr.V, maps, rp, l, stream);
        if (pr.bits == 4 && pr.gs == 128) return qmv::launch_b4g128_ringv(pr.V, maps, rp, l, stream);
        if (pr.bits == 2 && pr.gs == 64) return qmv::launch_b2g64_ringv(pr.V, maps, rp, l, stream);
        return qmv::launch_b2g128_ringv(pr.V, maps, rp, l, stream);
    }
    if (pr.V == 1 && pr.unit_mode == kUnitOne) {
        if (pr.bits == 4 && pr.gs == 64) return qmv::launch_b4g64_one(p, l, stream);
        if (pr.bits == 4 && pr.gs == 128) return qmv::launch_b4g128_one(p, l, stream);
        if (pr.bits == 2 && pr.gs == 64) return qmv::launch_b2g64_one(p, l, stream);
        return qmv::launch_b2g128_one(p, l, stream);
    }
    if (pr.V == 1) {
        qmv::RingParams rp;
        static_cast<qmv::Params &>(rp) = p;
        rp.uc = pr.uc; rp.unit_mode = pr.unit_mode; rp.pitch = pr.pitch; rp.sb_mode_unit = pr.sb_mode_unit;
        rp.sbox = pr.sbox; rp.slots = pr.slots; rp.consumers = pr.consumers;
        if (pr.bits == 4 && pr.gs == 64) return qmv::launch_b4g64_m1(maps, rp, l, stream);
        if (pr.bits == 4 && pr.gs == 128) return qmv::launch_b4g128_m1(maps, rp, l, stream);
        if (pr.bits == 2 && pr.gs == 64) return qmv::launch_b2g64_m1(maps, rp, l, stream);
        return qmv::launch_b2g128_m1(maps, rp, l, stream);
    }
    if (pr.bits == 4 && pr.gs == 64) return qmv::launch_b4g64_streamed(pr.V, p, l, stream);
    if (pr.bits == 4 && pr.gs == 128) return qmv::launch_b4g128_streamed(pr.V, p, l, stream);
    if (pr.bits == 2 && pr.gs == 64) return qmv::launch_b2g64_streamed(pr.V, p, l, stream);
    return qmv::launch_b2g128_streamed(pr.V, p, l, stream);
}

}  // namespace

namespace qmv {

// The host-side argument checks of a qmv_run_ex call, in the order they are
// reported: pointers, shape, flags, alignment.
qmv_status check_run_args(const void *w_q, const void *scales, const void *biases, const void *x, const void *y,
                          int M, int N, int K, int bits, int gs, const void *workspace, unsigned flags)
{
    const bool sb_packed = (flags & QMV_SB_INTERLEAVED) != 0;
    if (!w_q || !scales || (!biases && !sb_packed) || !x || !y) return QMV_ERR_NULL;
    qmv_status st = check_shape(M, N, K, bits, gs, true);
    if (st != QMV_OK) return st;
    if (flags & ~(QMV_F32_OUT | QMV_FORCE_M1_PER_COLUMN | QMV_PDL | QMV_SB_INTERLEAVED)) return QMV_ERR_FLAGS;
    const bool f32_out = (flags & QMV_F32_OUT) != 0;
    if (!aligned(w_q, 16) || !aligned(x, 16) || !aligned(scales, 16) || (!sb_packed && !aligned(biases, 16)) ||
        !aligned(y, f32_out ? 4 : 2) || (workspace && !aligned(workspace, 16)))
        return QMV_ERR_ALIGN;
    return QMV_OK;
}

qmv_status record_cuda_failure(const char *what, cudaError_t e) { return cuda_fail(what, e); }

}  // namespace qmv

namespace {

qmv_status run_impl(const uint32_t *w_q, const uint16_t *scales, const uint16_t *biases, const uint16_t *x, void *y,
                    int M, int N, int K, int bits, int gs, void *workspace, size_t workspace_bytes, unsigned flags,
                    cudaStream_t stream)
{
    qmv_status st = qmv::check_run_args(w_q, scales, biases, x, y, M, N, K, bits, gs, workspace, flags);
    if (st != QMV_OK) return st;
    const bool sb_packed = (flags & QMV_SB_INTERLEAVED) != 0;
    const bool f32_out = (flags & QMV_F32_OUT) != 0;

    static_assert(qmv::kMaxM == QMV_TILE_M, "launch width");
    // Vectors go through in launches of at most kMaxM (one each with
    // QMV_FORCE_M1_PER_COLUMN); a column's arithmetic does not depend on
    // which launch carries it, nor on how many vectors share that launch.
    const int tile = (flags & QMV_FORCE_M1_PER_COLUMN) != 0 ? 1 : qmv::kMaxM;

    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail("cudaGetDevice", ce);
    if (dev >= kMaxDevices) return cuda_fail("device index >= 64", cudaErrorInvalidDevice);
    int sms = 0;
    st = sm_count(dev, &sms);
    if (st != QMV_OK) return st;
    // at most two launch widths: full tiles and the remainder
    const int v_full = M < tile ? M : tile, v_rest = M > tile ? M % tile : 0;
    const Problem pr_full = plan(v_full, N, K, bits, gs, sms, sb_packed);
    const Problem pr_rest = v_rest ? plan(v_rest, N, K, bits, gs, sms, sb_packed) : pr_full;
    if (pr_full.smem > kSmemBudget || pr_rest.smem > kSmemBudget) {  // only a tuning override can get here
        snprintf(g_last_error, sizeof g_last_error, "launch plan needs %d bytes of shared memory",
                 pr_full.smem > pr_rest.smem ? pr_full.smem : pr_rest.smem);
        return QMV_ERR_CUDA;
    }
    const size_t need_full = workspace_bytes_for(pr_full), need_rest = workspace_bytes_for(pr_rest);
    const size_t need = need_full > need_rest ? need_full : need_rest;
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

    const bool pdl = (flags & QMV_PDL) != 0;
    const size_t ysize = f32_out ? sizeof(float) : sizeof(uint16_t);
    for (int pass = 0; pass < 2; ++pass) {
        const Problem &pr = pass == 0 ? pr_full : pr_rest;
        const int V = pass == 0 ? v_full : v_rest;
        const int m_lo = pass == 0 ? 0 : M - v_rest;
        const int m_hi = pass == 0 ? M - v_rest : M;
        if (V == 0 || m_lo >= m_hi) continue;

        qmv::RingMaps maps;
        memset(&maps, 0, sizeof maps);
        if ((V == 1 && pr.unit_mode != kUnitOne) || pr.ringv) {
            int enc = encode_sb_map(&maps.s, scales, pr);
            if (enc == 0 && !sb_packed) enc = encode_sb_map(&maps.b, biases, pr);
            if (enc == 0 && pr.unit_mode == qmv::kUnitTiles) enc = encode_w_map(&maps.w, w_q, pr);
            if (enc != 0) {
                snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled returned %d%s", enc,
                         enc < 0 ? " (driver entry point not found)" : "");
                return QMV_ERR_CUDA;
            }
        }

        qmv::Params p;
        p.err = err;
        p.w = reinterpret_cast<const uint8_t *>(w_q);
        p.scales = scales;
        p.biases = biases;
        p.N = N; p.K = K; p.G = pr.G; p.S_row = pr.S_row; p.ks = pr.ks; p.row_bytes = pr.row_bytes;
        p.NB = pr.NB; p.grid_rows = pr.grid_rows; p.cpc = pr.cpc; p.max_rb = pr.max_rb;
        p.f32_out = f32_out ? 1 : 0;
        p.sb_packed = sb_packed ? 1 : 0;
        p.early_weights = pdl ? 1 : 0;
        const bool split = split_bytes(pr) > 0;
        p.counters = split ? static_cast<unsigned *>(workspace) : nullptr;
        p.partials = split ? reinterpret_cast<float *>(static_cast<char *>(workspace) + counter_bytes(pr.NB)) : nullptr;
        p.xs_staged = V >= 2 ? static_cast<const uint8_t *>(workspace) + staged_offset(pr) : nullptr;
        for (int m = m_lo; m < m_hi; m += V) {
            p.x = x + size_t(m) * K;
            p.y = static_cast<char *>(y) + size_t(m) * N * ysize;
            ce = dispatch(pr, maps, p, pdl, stream);
            if (ce != cudaSuccess) return cuda_fail("kernel launch", ce);
        }
    }
    return QMV_OK;
}

}  // namespace

extern "C" int qmv_split_count(int N, int K, int bits, int group_size)
{
    if (check_shape(1, N, K, bits, group_size, false) != QMV_OK) return 0;
    return qmv::chunk_count(K);
}


extern "C" size_t qmv_workspace_size(int M, int N, int K, int bits, int group_size)
{
    if (check_shape(M, N, K, bits, group_size, true) != QMV_OK) return 0;
    // launches of kMaxM vectors and one of the remainder (see run_impl)
    const size_t full = workspace_bytes_for(plan(M < qmv::kMaxM ? M : qmv::kMaxM, N, K, bits, group_size, 0));
    const size_t rest = M > qmv::kMaxM && M % qmv::kMaxM ? workspace_bytes_for(plan(M % qmv::kMaxM, N, K, bits, group_size, 0)) : 0;
    return full > rest ? full : rest;
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

extern "C" qmv_status qmv_mxfp4_run(const uint32_t *w_q, const uint8_t *scales, const uint16_t *x, void *y, int M,
                                    int N, int K, unsigned flags, qmv_stream_t stream)
{
    if (!w_q || !scales || !x || !y) return QMV_ERR_NULL;
    if (N < 1 || N > (1 << 30) || K < 1 || K % 32 != 0 || K > (1 << 24) || (long long)N * (K / 32) >= (1ll << 31))
        return QMV_ERR_SHAPE;
    if (M < 1 || M > QMV_MAX_M) return QMV_ERR_M_RANGE;
    if (flags & ~(QMV_F32_OUT | QMV_FORCE_M1_PER_COLUMN)) return QMV_ERR_FLAGS;
    const bool f32_out = (flags & QMV_F32_OUT) != 0;
    if (!aligned(w_q, 16) || !aligned(x, 16) || !aligned(y, f32_out ? 4 : 2)) return QMV_ERR_ALIGN;

    // launches of QMV_TILE_M vectors (one each with QMV_FORCE_M1_PER_COLUMN);
    // a column's arithmetic does not depend on its launch's width
    const int tile = (flags & QMV_FORCE_M1_PER_COLUMN) != 0 ? 1 : QMV_TILE_M;
    const size_t ysize = f32_out ? sizeof(float) : sizeof(uint16_t);
    qmv::MxParams p;
    p.w = w_q;
    p.scales = scales;
    p.N = N;
    p.K = K;
    p.f32_out = f32_out ? 1 : 0;
    for (int m = 0; m < M; m += tile) {
        const int V = M - m < tile ? M - m : tile;
        p.x = x + size_t(m) * K;
        p.y = static_cast<char *>(y) + size_t(m) * N * ysize;
        const cudaError_t ce = qmv::launch_mxfp4(V, p, reinterpret_cast<cudaStream_t>(stream));
        if (ce != cudaSuccess) return cuda_fail("mxfp4 kernel launch", ce);
    }
    return QMV_OK;
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
        case QMV_ERR_M_RANGE: return "QMV_ERR_M_RANGE: M must be in [1, 256]";
        case QMV_ERR_ALIGN: return "QMV_ERR_ALIGN: w_q, x, scales, biases and workspace need 16-byte alignment, y 2 (f32 y: 4)";
        case QMV_ERR_CUDA: return "QMV_ERR_CUDA: a CUDA runtime call or kernel launch failed";
        case QMV_ERR_WORKSPACE: return "QMV_ERR_WORKSPACE: workspace smaller than qmv_workspace_size()";
        case QMV_ERR_VALUE: return "QMV_ERR_VALUE: a quantized value does not fit in `bits` bits";
        case QMV_ERR_FLAGS: return "QMV_ERR_FLAGS: unknown flag bits";
    }
    return "unknown qmv_status";
}
