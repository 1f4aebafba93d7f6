// The mxfp4 mode of qmv: y = W x with E2M1 weights and one E8M0 scale per 32
// consecutive weights along K.
//
// mlxcel issue #1289, section "Scope limits, stated honestly", names the fp
// modes (mxfp4) as the second phase of the order-preserving streamed qmv and
// gives no format; the reading taken is the OCP MX v1.0 MXFP4 format: an E2M1
// element has a sign (bit 3), a 2-bit exponent with bias 1 (bits 2..1) and one
// mantissa bit (bit 0), exponent field 0 being subnormal; an E8M0 scale byte e
// is 2^(e - 127), e = 255 being NaN. The codes are packed like the affine
// 4-bit fields: element k of a row at bits [4 (k % 8), 4 (k % 8) + 4) of word
// k / 8, so the 32 codes of one scale block are one aligned 16-byte vector.
//
// One kernel template serves every launch width V = 1..16, and an output's
// fp32 operation sequence is the same for every V, so every column of a
// V-vector launch is bit-identical to the one-vector launch on that column
// (issue #1289, "The observation this rests on"). For row n and vector m:
//
//   1. block b (32 elements): an even chain and an odd chain, each
//      a = fma(v_i, x_i, a) from +0 in increasing i (both products exact in
//      fp32: v has two significant bits, x eight), then d_b = a_even + a_odd
//      and t_b = d_b * 2^(e_b - 127);
//   2. lane l of the row's warp folds the blocks b = l, l + 32, l + 64, ...
//      in increasing order: p_l = (((+0 + t_l) + t_{l+32}) + ...);
//   3. y = p_0 + ... + p_31 by the xor butterfly over offsets 16, 8, 4, 2, 1,
//      then one rounding to bf16 (nearest even), or the fp32 value itself.
//
// The elements come out of the codes by the E2M1 -> f16x2 conversion of
// sm_100-class parts (two elements per instruction, exact) and one exact
// f16 -> f32 widening each; the two chains run as one packed fma.rn.f32x2.
//
// A CTA holds 4 warps of 4 rows each. K goes by in chunks of 1024 elements,
// one 32-block per lane; each chunk of x is staged once per CTA into shared
// memory as fp32 pairs laid out [vector][pair / 2][lane][pair % 2] (a warp's
// reads of two pairs cover 512 contiguous bytes), and every x pair read serves the
// warp's 4 rows. Up to 4 vectors: all of them are staged per chunk, a chunk's
// weights convert once per pass of up to 4 vectors, and (2..4 vectors) the
// next chunk's weights are loaded while the current one is computed. From 5
// vectors on, the vectors go in passes of at most 5 outermost, each over all
// of K with its partials in registers (mx_pass), so a chunk's weights convert
// once per pass and a CTA needs at most 20 KB of shared memory: four CTAs (16
// warps) share an SM. 16 rows a CTA keep the last wave short: a 15360-row
// matrix is 960 CTAs, 6.3 per SM (with 32 rows a CTA, 3.2 per SM, the last
// of them ran on a half-empty GPU).
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "qmv_launch_decl.h"

namespace qmv {
namespace {

constexpr int kMxWarps = 4;
constexpr int kMxRows = 4;                         // rows per warp
constexpr int kMxRowsPerCta = kMxWarps * kMxRows;  // 16
constexpr int kMxChunk = 32 * 32;                  // elements per K-chunk: one 32-block per lane
constexpr int kMxPairs = 16;                       // element pairs per block
constexpr int kMxPass = 4;                         // vectors per pass over a chunk's weights

// Eight E2M1 codes (one 32-bit word, element 2j in the low nibble of byte j)
// to four f16x2 words, word j holding elements 2j (low half) and 2j + 1.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4])
{
    asm("{\n\t"
        ".reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t"
        "}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// f16x2 -> a pair of fp32 in one 64-bit register (low half = low element).
__device__ __forceinline__ uint64_t f16x2_to_f32x2(uint32_t h)
{
    uint64_t d;
    asm("{\n\t"
        ".reg .f16 lo, hi;\n\t"
        ".reg .f32 a, b;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "cvt.f32.f16 a, lo;\n\t"
        "cvt.f32.f16 b, hi;\n\t"
        "mov.b64 %0, {a, b};\n\t"
        "}"
        : "=l"(d)
        : "r"(h));
    return d;
}

__device__ __forceinline__ uint64_t mx_ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// E8M0 byte -> 2^(e - 127) as fp32 (e = 0 is the subnormal 2^-127; 255 is NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e)
{
    const uint32_t bits = e == 0u ? 0x00400000u : (e == 255u ? 0x7fc00000u : e << 23);
    return __uint_as_float(bits);
}

// Staged x of a chunk: pair i (elements 32 l + 2 i, 32 l + 2 i + 1) of vector
// v for lane l, laid out [v][i / 2][l][i % 2], so that a lane's pairs 2j and
// 2j + 1 are one 16-byte vector and a warp's read of one pair is 16 bytes a
// lane apart (two of the warp's reads cover 512 contiguous bytes).
__device__ __forceinline__ int mx_x_index(int v, int i, int lane)
{
    return ((v * (kMxPairs / 2) + (i >> 1)) * 32 + lane) * 2 + (i & 1);
}

// Stages x[v][k0 .. k0 + kn) for v < V into xs at mx_x_index as fp32 pairs
// (element 2i of block l in the low half). kn is a multiple of 32. Thread
// item t of a vector takes the 8 elements (t / 32) * 8 .. + 7 of block t % 32,
// so the 32 threads of a warp write the same pair of 32 consecutive lanes.
template <int V>
__device__ __forceinline__ void mx_stage_chunk(uint64_t *xs, const uint16_t *x, int K, int k0, int kn)
{
    for (int item = threadIdx.x; item < V * (kMxChunk / 8); item += kMxWarps * 32) {
        const int v = item / (kMxChunk / 8);
        const int blk = item % 32, quad = (item % (kMxChunk / 8)) / 32;
        const int e0 = blk * 32 + quad * 8;
        if (e0 >= kn) continue;
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(x + size_t(v) * K + k0 + e0));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            xs[mx_x_index(v, quad * 4 + q, blk)] = (uint64_t(w[q] & 0xffff0000u) << 32) | uint64_t(w[q] << 16);
    }
}

// CTAs per SM the register budget must allow: eight for one vector (at most
// 64 registers), so that a 15360-row matrix (960 CTAs) runs as one wave on
// 152 SMs; four otherwise (at most 128 registers, 16 warps per SM).
template <int V>
constexpr int mx_min_blocks() { return V == 1 ? 8 : 4; }

// Several vectors (V >= 5): the vectors go in passes of at most kMxWidePass,
// each pass running over all of K, so that a pass's partials stay in
// registers and the chunk's x is staged for the pass's vectors only. Each
// pass re-reads the warp's weights, which the first pass has just brought
// into L2. Vectors [v0, v0 + VPN) of the warp's rows, steps 1-4.
constexpr int kMxWidePass = 5;

template <int VPN>
__device__ __forceinline__ void mx_pass(const MxParams &p, uint64_t *xs, int v0, int row0, int nlive, int lane)
{
    const int B = p.K >> 5;
    const int nchunks = (B + 31) >> 5;
    const uint4 *wbase = reinterpret_cast<const uint4 *>(p.w) + size_t(row0) * B;
    const uint8_t *sbase = p.scales + size_t(row0) * B;
    const uint16_t *xv = p.x + size_t(v0) * p.K;

    float part[VPN][kMxRows];
#pragma unroll
    for (int v = 0; v < VPN; ++v)
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) part[v][r] = 0.0f;

#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
        const int k0 = c * kMxChunk;
        const int kn = p.K - k0 < kMxChunk ? p.K - k0 : kMxChunk;
        const int b = c * 32 + lane;
        uint4 wc[kMxRows];
        uint32_t sc[kMxRows];
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) {
            const bool ok = r < nlive && b < B;
            wc[r] = ok ? __ldg(wbase + size_t(r) * B + b) : make_uint4(0u, 0u, 0u, 0u);
            sc[r] = ok ? __ldg(sbase + size_t(r) * B + b) : 0u;
        }
        __syncthreads();  // every warp is done reading the previous chunk of x
        mx_stage_chunk<VPN>(xs, xv, p.K, k0, kn);
        __syncthreads();
        if (b < B) {
            uint64_t acc[VPN][kMxRows];
#pragma unroll
            for (int v = 0; v < VPN; ++v)
#pragma unroll
                for (int r = 0; r < kMxRows; ++r) acc[v][r] = 0ull;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t h[kMxRows][4];
#pragma unroll
                for (int r = 0; r < kMxRows; ++r) {
                    const uint32_t word = j == 0 ? wc[r].x : j == 1 ? wc[r].y : j == 2 ? wc[r].z : wc[r].w;
                    e2m1x8_to_f16x2(word, h[r]);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = 4 * j + k;
                    uint64_t wv[kMxRows];
#pragma unroll
                    for (int r = 0; r < kMxRows; ++r) wv[r] = f16x2_to_f32x2(h[r][k]);
#pragma unroll
                    for (int v = 0; v < VPN; ++v) {
                        const uint64_t x2 = xs[mx_x_index(v, i, lane)];
#pragma unroll
                        for (int r = 0; r < kMxRows; ++r) acc[v][r] = mx_ffma2(wv[r], x2, acc[v][r]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kMxRows; ++r) {
                const float scale = e8m0_to_f32(sc[r]);
#pragma unroll
                for (int v = 0; v < VPN; ++v) {
                    const float ae = __uint_as_float(uint32_t(acc[v][r]));
                    const float ao = __uint_as_float(uint32_t(acc[v][r] >> 32));
                    part[v][r] = __fadd_rn(part[v][r], __fmul_rn(__fadd_rn(ae, ao), scale));
                }
            }
        }
    }
    // butterfly over the lanes: every lane ends with the same sum
#pragma unroll
    for (int v = 0; v < VPN; ++v)
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) {
            float sum = part[v][r];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, off));
            part[v][r] = sum;
        }
#pragma unroll
    for (int r = 0; r < kMxRows; ++r) {
        if (lane != r || r >= nlive) continue;
        const size_t n = size_t(row0 + r);
#pragma unroll
        for (int v = 0; v < VPN; ++v) {
            if (p.f32_out)
                static_cast<float *>(p.y)[size_t(v0 + v) * p.N + n] = part[v][r];
            else
                static_cast<__nv_bfloat16 *>(p.y)[size_t(v0 + v) * p.N + n] = __float2bfloat16_rn(part[v][r]);
        }
    }
}

// Pass structure of a V-vector launch with V >= 5: passes of VP vectors, the
// last one of the remainder.
template <int V>
struct MxPasses {
    static constexpr int N = (V + kMxWidePass - 1) / kMxWidePass;
    static constexpr int VP = (V + N - 1) / N;
    static constexpr int LAST = V - (N - 1) * VP;
};

template <int V>
__device__ __forceinline__ void qmv_mxfp4_narrow(MxParams p);

template <int V>
__global__ void __launch_bounds__(kMxWarps * 32, mx_min_blocks<V>()) qmv_mxfp4(MxParams p)
{
    if constexpr (V >= 5) {
        extern __shared__ __align__(16) uint64_t mx_xs[];  // VP vectors of staged x (mx_x_index)
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const int row0 = blockIdx.x * kMxRowsPerCta + warp * kMxRows;
        const int nlive = p.N - row0;
        using PS = MxPasses<V>;
#pragma unroll 1
        for (int ps = 0; ps + 1 < PS::N; ++ps) mx_pass<PS::VP>(p, mx_xs, ps * PS::VP, row0, nlive, lane);
        mx_pass<PS::LAST>(p, mx_xs, (PS::N - 1) * PS::VP, row0, nlive, lane);
        return;
    } else {
        qmv_mxfp4_narrow<V>(p);
    }
}

template <int V>
__device__ __forceinline__ void qmv_mxfp4_narrow(MxParams p)
{
    extern __shared__ __align__(16) uint64_t mx_xs[];  // V vectors of staged x (mx_x_index)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row0 = blockIdx.x * kMxRowsPerCta + warp * kMxRows;
    const int B = p.K >> 5;  // scale blocks per row
    const int nchunks = (B + 31) >> 5;

    // rows row0 .. row0 + nlive - 1 exist; one 16-byte vector of codes per block
    const int nlive = p.N - row0;
    const uint4 *wbase = reinterpret_cast<const uint4 *>(p.w) + size_t(row0) * B;
    const uint8_t *sbase = p.scales + size_t(row0) * B;

    float part[V][kMxRows];
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) part[v][r] = 0.0f;

    // The codes and scale bytes of block b for the warp's rows.
    auto load_block = [&](int b, uint4 (&w)[kMxRows], uint32_t (&sv)[kMxRows]) {
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) {
            const bool ok = r < nlive && b < B;
            w[r] = ok ? __ldg(wbase + size_t(r) * B + b) : make_uint4(0u, 0u, 0u, 0u);
            sv[r] = ok ? __ldg(sbase + size_t(r) * B + b) : 0u;
        }
    };
    // Several vectors: the next chunk's loads are issued a chunk ahead. One
    // vector: a chunk's loads are issued before its x is staged; the eight CTAs
    // an SM then holds keep enough of them in flight, and the 64-register
    // budget has no room for a second set.
    constexpr bool kAhead = V > 1;
    uint4 wc[kMxRows];
    uint32_t sc[kMxRows];
    if (kAhead) load_block(lane, wc, sc);

    for (int c = 0; c < nchunks; ++c) {
        const int k0 = c * kMxChunk;
        const int kn = p.K - k0 < kMxChunk ? p.K - k0 : kMxChunk;
        if (!kAhead) load_block(c * 32 + lane, wc, sc);
        __syncthreads();  // every warp is done reading the previous chunk of x
        mx_stage_chunk<V>(mx_xs, p.x, p.K, k0, kn);
        __syncthreads();

        uint4 wn[kMxRows];
        uint32_t sn[kMxRows];
        if (kAhead) load_block((c + 1) * 32 + lane, wn, sn);

        if (c * 32 + lane < B) {
            float scale[kMxRows];
#pragma unroll
            for (int r = 0; r < kMxRows; ++r) scale[r] = e8m0_to_f32(sc[r]);
#pragma unroll
            for (int v0 = 0; v0 < V; v0 += kMxPass) {
                uint64_t acc[kMxPass][kMxRows];
#pragma unroll
                for (int v = 0; v < kMxPass; ++v)
#pragma unroll
                    for (int r = 0; r < kMxRows; ++r) acc[v][r] = 0ull;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t h[kMxRows][4];
#pragma unroll
                    for (int r = 0; r < kMxRows; ++r) {
                        const uint32_t word = j == 0 ? wc[r].x : j == 1 ? wc[r].y : j == 2 ? wc[r].z : wc[r].w;
                        e2m1x8_to_f16x2(word, h[r]);
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int i = 4 * j + k;
                        uint64_t wv[kMxRows];
#pragma unroll
                        for (int r = 0; r < kMxRows; ++r) wv[r] = f16x2_to_f32x2(h[r][k]);
#pragma unroll
                        for (int v = 0; v < kMxPass; ++v) {
                            if (v0 + v >= V) continue;
                            const uint64_t xv = mx_xs[mx_x_index(v0 + v, i, lane)];
#pragma unroll
                            for (int r = 0; r < kMxRows; ++r) acc[v][r] = mx_ffma2(wv[r], xv, acc[v][r]);
                        }
                    }
                }
#pragma unroll
                for (int v = 0; v < kMxPass; ++v) {
                    if (v0 + v >= V) continue;
#pragma unroll
                    for (int r = 0; r < kMxRows; ++r) {
                        const float ae = __uint_as_float(uint32_t(acc[v][r]));
                        const float ao = __uint_as_float(uint32_t(acc[v][r] >> 32));
                        const float t = __fmul_rn(__fadd_rn(ae, ao), scale[r]);
                        part[v0 + v][r] = __fadd_rn(part[v0 + v][r], t);
                    }
                }
            }
        }
        if (kAhead) {
#pragma unroll
            for (int r = 0; r < kMxRows; ++r) {
                wc[r] = wn[r];
                sc[r] = sn[r];
            }
        }
    }

    // butterfly over the lanes: every lane ends with the same sum
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
        for (int r = 0; r < kMxRows; ++r) {
            float s = part[v][r];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
            part[v][r] = s;
        }
#pragma unroll
    for (int r = 0; r < kMxRows; ++r) {
        if (lane != r || r >= nlive) continue;
        const size_t n = size_t(row0 + r);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            if (p.f32_out)
                static_cast<float *>(p.y)[size_t(v) * p.N + n] = part[v][r];
            else
                static_cast<__nv_bfloat16 *>(p.y)[size_t(v) * p.N + n] = __float2bfloat16_rn(part[v][r]);
        }
    }
}

template <int V>
cudaError_t launch_mx_v(const MxParams &p, cudaStream_t stream)
{
    // The opt-in dynamic shared-memory limit is a per-device kernel attribute;
    // raise it (never lower it) under a lock the first time a device needs it.
    static std::atomic<int> configured[64] = {};
    // staged x: the launch's vectors, or (V >= 5) one pass's
    constexpr int VS = V >= 5 ? MxPasses<V >= 5 ? V : 5>::VP : V;
    const int smem = VS * kMxPairs * 32 * int(sizeof(uint64_t));
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    if (configured[dev].load() < smem) {
        static std::mutex m;
        std::lock_guard<std::mutex> lock(m);
        if (configured[dev].load() < smem) {
            e = cudaFuncSetAttribute(qmv_mxfp4<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            configured[dev].store(smem);
        }
    }
    const unsigned grid = unsigned((p.N + kMxRowsPerCta - 1) / kMxRowsPerCta);
    qmv_mxfp4<V><<<grid, kMxWarps * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mxfp4(int V, const MxParams &p, cudaStream_t stream)
{
    switch (V) {
#define QMV_MX_CASE(v) \
    case v: return launch_mx_v<v>(p, stream);
        QMV_MX_CASE(1) QMV_MX_CASE(2) QMV_MX_CASE(3) QMV_MX_CASE(4) QMV_MX_CASE(5) QMV_MX_CASE(6)
        QMV_MX_CASE(7) QMV_MX_CASE(8) QMV_MX_CASE(9) QMV_MX_CASE(10) QMV_MX_CASE(11) QMV_MX_CASE(12)
        QMV_MX_CASE(13) QMV_MX_CASE(14) QMV_MX_CASE(15) QMV_MX_CASE(16)
#undef QMV_MX_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmv
