// sm_103a kernels of the affine group-quantized mat-vec:
//
//   y[m, n] = sum_g ( s[n,g] * sum_{i in g} q[n,i] x[m,i] + b[n,g] * sum_{i in g} x[m,i] )
//
// the factored group dot of mlxcel issue #1289 ("Correction to the obvious
// sketch": scale * accum + sum * bias, no dequantized weight) applied once per
// group (mlxcel PR #1681, "Not covered"), and its order-preserving streamed
// form (#1289 "Step 2"): the weights are read and decoded once and reused for
// V <= 16 activation vectors, with each vector's fp32 operation sequence
// exactly the one an M = 1 launch performs.
//
// Work decomposition (nothing here depends on V):
//  * CTA = 8 warps = 64 consecutive output rows x one K-split (blockIdx.y).
//  * A warp owns 8 rows. Its lane (p, j), p = lane/8, j = lane%8, owns the row
//    pair {p, p+4} and slice j: local group 8*t + j of the split in stage t.
//  * Weights stream through a private ring per warp: 128-byte x 8-row TMA
//    boxes, 128B-swizzled, one mbarrier per stage; the warp is its own
//    producer (lane 0 refills a slot after the warp has read it).
//  * x is staged once per CTA into shared memory as fp32, pre-multiplied by
//    2^(-bits * (i mod 16/bits)), with a 16-byte pad after each group so the
//    eight slices read eight different bank groups; sum(x) per group is
//    staged beside it.
//
// Fixed fp32 order for output (m, n) -- the definition the bit-identity rests on:
//  1. per group: two running sums, even and odd elements, each in increasing
//     element order: a_e = fma(q_t, x_t, a_e) (t even), a_o likewise (t odd),
//     starting from +0 (a packed fma.rn.f32x2); d = a_e + a_o.
//     Products q_t * x_t are exact in fp32 (4-bit integer times 8-bit mantissa).
//  2. fold: P = fma(s_g, d, P); P = fma(b_g, sx_g, P), where P is the running
//     value of slice j over its groups j, j+8, j+16, ... in increasing order
//     and sx_g = (((x_0 + x_1) + x_2) + ...) over the group.
//  3. slices: butterfly over j with xor 4, 2, 1 (each step P + P').
//  4. splits: y = ((p_0 + p_1) + p_2) + ... in split order (one split: y = p_0).
//  5. y rounded once to bf16, nearest even.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qmv_plan.h"

namespace qmv {

// ------------------------------------------------------------ PTX helpers --

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: gives up after ~2 s of wall time or 2^28 polls, whichever
// comes first, so a lost transfer can never hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1; it < (1u << 28); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > 2000000000ull) return false;
    }
    return false;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2-D TMA tile load (global -> this CTA's shared memory), completion counted
// in bytes on `bar`. x is the byte column, y the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h)
{
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// ------------------------------------------------------ field extraction --

// binary32 2^23: OR-ing an integer m < 2^23 into its significand gives 2^23 + m.
constexpr uint32_t kMagic = 0x4B000000u;

__device__ __forceinline__ float2 magic_pair(uint32_t w, uint32_t mask_lo, uint32_t mask_hi)
{
    return make_float2(__uint_as_float((w & mask_lo) | kMagic), __uint_as_float((w & mask_hi) | kMagic));
}

// Element pairs (2p, 2p+1) of one packed word, as exact floats q * 2^(bits*k),
// k the element's position inside its 16-bit half. The matching x values were
// staged pre-multiplied by 2^(-bits*k), so each product equals q * x exactly.
template <int BITS>
__device__ __forceinline__ void extract_pairs(uint32_t w, float2 (&q)[16 / BITS])
{
    const float2 neg_magic = make_float2(-8388608.0f, -8388608.0f);
    const uint32_t lo = w, hi = w >> 16;
    if constexpr (BITS == 4) {
        q[0] = __fadd2_rn(magic_pair(lo, 0x000Fu, 0x00F0u), neg_magic);
        q[1] = __fadd2_rn(magic_pair(lo, 0x0F00u, 0xF000u), neg_magic);
        q[2] = __fadd2_rn(magic_pair(hi, 0x000Fu, 0x00F0u), neg_magic);
        q[3] = __fadd2_rn(magic_pair(hi, 0x0F00u, 0xF000u), neg_magic);
    } else {
        q[0] = __fadd2_rn(magic_pair(lo, 0x0003u, 0x000Cu), neg_magic);
        q[1] = __fadd2_rn(magic_pair(lo, 0x0030u, 0x00C0u), neg_magic);
        q[2] = __fadd2_rn(magic_pair(lo, 0x0300u, 0x0C00u), neg_magic);
        q[3] = __fadd2_rn(magic_pair(lo, 0x3000u, 0xC000u), neg_magic);
        q[4] = __fadd2_rn(magic_pair(hi, 0x0003u, 0x000Cu), neg_magic);
        q[5] = __fadd2_rn(magic_pair(hi, 0x0030u, 0x00C0u), neg_magic);
        q[6] = __fadd2_rn(magic_pair(hi, 0x0300u, 0x0C00u), neg_magic);
        q[7] = __fadd2_rn(magic_pair(hi, 0x3000u, 0xC000u), neg_magic);
    }
}

__device__ __forceinline__ uint32_t word_of(const uint4 &c, int k)
{
    return k == 0 ? c.x : (k == 1 ? c.y : (k == 2 ? c.z : c.w));
}

// ----------------------------------------------------------- group dot --

// Address of 16-byte chunk c of warp-local row r inside a 128B-swizzled box.
__device__ __forceinline__ const uint4 *box_chunk(const uint8_t *box, int r, int c)
{
    return reinterpret_cast<const uint4 *>(box + r * kBoxBytes + ((c ^ (r & 7)) << 4));
}

// One group of the lane's two rows against V staged vectors: step 1 of the
// fixed order. acc[r][v] = (a_e, a_o).
template <int BITS, int GS, int V>
__device__ __forceinline__ void group_dot(const uint8_t *stage, int j, int rA, int rB, const float *xg,
                                          int xvstride, float2 (&acc)[2][V])
{
    constexpr int kGB = group_bytes(BITS, GS);
    constexpr int kChunks = kGB / 16;
    constexpr int kGPB = groups_per_box(BITS, GS);
    constexpr int kPerWord = 32 / BITS;
    const uint8_t *box = stage + (j / kGPB) * kBoxSmem;
    const int c0 = (j % kGPB) * kChunks;

    uint4 wa[kChunks], wb[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        wa[c] = *box_chunk(box, rA, c0 + c);
        wb[c] = *box_chunk(box, rB, c0 + c);
    }
#pragma unroll
    for (int v = 0; v < V; ++v) {
        acc[0][v] = make_float2(0.0f, 0.0f);
        acc[1][v] = make_float2(0.0f, 0.0f);
    }
#pragma unroll
    for (int w = 0; w < kChunks * 4; ++w) {
        float2 qa[kPerWord / 2], qb[kPerWord / 2];
        extract_pairs<BITS>(word_of(wa[w / 4], w % 4), qa);
        extract_pairs<BITS>(word_of(wb[w / 4], w % 4), qb);
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const float4 *xv = reinterpret_cast<const float4 *>(xg + v * xvstride + w * kPerWord);
#pragma unroll
            for (int h = 0; h < kPerWord / 4; ++h) {
                const float4 x4 = xv[h];
                const float2 x01 = make_float2(x4.x, x4.y), x23 = make_float2(x4.z, x4.w);
                acc[0][v] = __ffma2_rn(qa[2 * h], x01, acc[0][v]);
                acc[1][v] = __ffma2_rn(qb[2 * h], x01, acc[1][v]);
                acc[0][v] = __ffma2_rn(qa[2 * h + 1], x23, acc[0][v]);
                acc[1][v] = __ffma2_rn(qb[2 * h + 1], x23, acc[1][v]);
            }
        }
    }
}

// ---------------------------------------------------------------- kernel --

// Position of a warp in its (tile, chunk, stage) sequence. Tiles advance by
// gridDim.x (persistent CTAs); chunks run over the CTA's chunk range.
struct Cursor {
    int tile, chunk, t;
};

// First group of chunk c (chunk boundaries are box-aligned; see split_count).
template <int BITS, int GS>
__device__ __forceinline__ int chunk_first_group(const Params &p, int c)
{
    const int g = (c * p.nbox / p.ks) * groups_per_box(BITS, GS);
    return g < p.G ? g : p.G;
}

template <int BITS, int GS, int V>
__device__ __forceinline__ void qmv_body(const CUtensorMap *tmap_w, const Params &p)
{
    constexpr int kGPB = groups_per_box(BITS, GS);
    constexpr int kBPS = boxes_per_stage(BITS, GS);
    constexpr int kStageBytes = stage_bytes(BITS, GS);
    constexpr int kStages = ring_stages(BITS, GS);
    constexpr int kXS = x_stride(GS);
    constexpr int kPerHalf = 16 / BITS;
    constexpr int kGB = group_bytes(BITS, GS);

    extern __shared__ uint8_t smem_raw[];
    __shared__ unsigned s_ticket;
    __shared__ int s_cg0[kMaxChunksPerCta + 1];  // first group of each chunk of this CTA, and the end
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemLayout L = smem_layout(BITS, GS, V, p.gsm);
    float *xs = reinterpret_cast<float *>(smem + L.xs);
    float *sxs = reinterpret_cast<float *>(smem + L.sx);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pr = lane >> 3, j = lane & 7;
    const int chunk_lo = blockIdx.y * p.cps;
    const int chunk_hi = chunk_lo + p.cps < p.ks ? chunk_lo + p.cps : p.ks;
    const int ncpc = chunk_hi - chunk_lo;  // chunks of this CTA (<= kMaxChunksPerCta, checked on the host)
    if (tid <= ncpc) s_cg0[tid] = chunk_first_group<BITS, GS>(p, chunk_lo + tid);
    __syncthreads();
    const int g_lo = s_cg0[0];
    const int gsn = s_cg0[ncpc] - g_lo;  // groups of x staged by this CTA
    // chunk-local helpers (c is relative to chunk_lo)
    auto cg0 = [&](int c) { return s_cg0[c]; };
    auto cstages = [&](int c) { return (s_cg0[c + 1] - s_cg0[c] + kSlices - 1) / kSlices; };

    const uint32_t bar0 = smem_u32(bars + warp * kStages);
    const uint32_t ring_w = smem_u32(smem + L.ring + warp * kRingBytesPerWarp);
    const uint64_t pol = l2_evict_first_policy();

    auto warp_row0 = [&](int tile) { return tile * kRowsPerCta + warp * kRowsPerWarp; };
    auto valid = [&](const Cursor &c) { return c.tile < p.ntiles && warp_row0(c.tile) < p.N; };
    auto advance = [&](Cursor &c) {
        if (++c.t == cstages(c.chunk)) {
            c.t = 0;
            if (++c.chunk == ncpc) {
                c.chunk = 0;
                c.tile += gridDim.x;
            }
        }
    };
    auto issue = [&](const Cursor &c, int slot) {
        const int gc0 = cg0(c.chunk), gc1 = cg0(c.chunk + 1);
        const int gl0 = gc0 + c.t * kSlices;
        int nb = (gc1 - gl0 + kGPB - 1) / kGPB;
        nb = nb < kBPS ? nb : kBPS;
        mbar_arrive_expect_tx(bar0 + 8 * slot, nb * kBoxSmem);
        for (int b = 0; b < nb; ++b)
            tma_load_2d(ring_w + slot * kStageBytes + b * kBoxSmem, tmap_w, gl0 * kGB + b * kBoxBytes,
                        warp_row0(c.tile), bar0 + 8 * slot, pol);
    };

    // Weight tiles first: they do not depend on x, so their latency overlaps the staging below.
    Cursor prod = {int(blockIdx.x), 0, 0};
    int issued = 0;
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
        for (; issued < kStages && valid(prod); ++issued, advance(prod)) issue(prod, issued);
    }
    __syncwarp();

    // Stage x for groups [g_lo, g_lo + gsn): fp32, position-scaled, 8 elements per task.
    {
        constexpr int kUPG = GS / 8;
        const int per_vec = gsn * kUPG, total = V * per_vec;
        for (int u0 = tid; u0 < total; u0 += 4 * kThreads) {
            uint4 raw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int u = u0 + k * kThreads;
                if (u < total) {
                    const int v = u / per_vec, rem = u - v * per_vec;
                    raw[k] = __ldg(reinterpret_cast<const uint4 *>(p.x + size_t(v) * p.K + size_t(g_lo) * GS) + rem);
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int u = u0 + k * kThreads;
                if (u < total) {
                    const int v = u / per_vec, rem = u - v * per_vec;
                    const int gl = rem / kUPG, e8 = rem - gl * kUPG;
                    const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
                    float f[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t bits = (i & 1) ? (w4[i / 2] & 0xFFFF0000u) : (w4[i / 2] << 16);
                        const float scale = __uint_as_float(uint32_t(127 - BITS * (i % kPerHalf)) << 23);
                        f[i] = __fmul_rn(__uint_as_float(bits), scale);
                    }
                    float4 *dst = reinterpret_cast<float4 *>(xs + (v * p.gsm + gl) * kXS + e8 * 8);
                    dst[0] = make_float4(f[0], f[1], f[2], f[3]);
                    dst[1] = make_float4(f[4], f[5], f[6], f[7]);
                }
            }
        }
        // sum(x) per (vector, group): eight sums of eight consecutive elements,
        // each left to right, then those eight (sixteen for gs=128) left to right.
        for (int idx = tid; idx < V * gsn; idx += kThreads) {
            const int v = idx / gsn, gl = idx - v * gsn;
            const uint4 *src = reinterpret_cast<const uint4 *>(p.x + size_t(v) * p.K + size_t(g_lo + gl) * GS);
            uint4 raw[kUPG];
#pragma unroll
            for (int k = 0; k < kUPG; ++k) raw[k] = __ldg(src + k);
            float total_sum = 0.0f;
#pragma unroll
            for (int k = 0; k < kUPG; ++k) {
                const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
                float s8 = __uint_as_float(w4[0] << 16);
#pragma unroll
                for (int i = 1; i < 8; ++i)
                    s8 = __fadd_rn(s8, __uint_as_float((i & 1) ? (w4[i / 2] & 0xFFFF0000u) : (w4[i / 2] << 16)));
                total_sum = k == 0 ? s8 : __fadd_rn(total_sum, s8);
            }
            sxs[v * p.gsm + gl] = total_sum;
        }
    }
    __syncthreads();

    auto store_y = [&](int v, int n, float val) {
        if (p.f32_out)
            static_cast<float *>(p.y)[size_t(v) * p.N + n] = val;
        else
            static_cast<__nv_bfloat16 *>(p.y)[size_t(v) * p.N + n] = __float2bfloat16_rn(val);
    };

    const int rA = pr, rB = pr + 4;
    int consumed = 0;
    bool ok = true;
    // Metadata (scale, bias) of the lane's group one stage ahead of the weights.
    Cursor meta = {int(blockIdx.x), 0, 0};
    uint16_t msA = 0, mbA = 0, msB = 0, mbB = 0;
    auto load_meta = [&](const Cursor &c) {
        if (!valid(c)) return;
        const int gc0 = cg0(c.chunk), gc1 = cg0(c.chunk + 1);
        int g = gc0 + c.t * kSlices + j;
        g = g < gc1 ? g : gc1 - 1;
        const int r0 = warp_row0(c.tile);
        const int nA = r0 + rA < p.N ? r0 + rA : p.N - 1;
        const int nB = r0 + rB < p.N ? r0 + rB : p.N - 1;
        msA = __ldg(p.scales + size_t(nA) * p.G + g);
        mbA = __ldg(p.biases + size_t(nA) * p.G + g);
        msB = __ldg(p.scales + size_t(nB) * p.G + g);
        mbB = __ldg(p.biases + size_t(nB) * p.G + g);
    };
    load_meta(meta);

    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x) {
        const int row0 = warp_row0(tile);
        const bool active = row0 < p.N;
        const int nA = row0 + rA, nB = row0 + rB;
        float yr[2][V];
        if (active && ok) {
            for (int c = 0; c < ncpc; ++c) {
                const int gc0 = cg0(c), gc1 = cg0(c + 1);
                const int nst = (gc1 - gc0 + kSlices - 1) / kSlices;
                float part[2][V];
#pragma unroll
                for (int v = 0; v < V; ++v) part[0][v] = part[1][v] = 0.0f;
                for (int t = 0; t < nst; ++t) {
                    const int slot = consumed % kStages;
                    const uint32_t parity = (consumed / kStages) & 1;
                    const float fsA = bf16_bits_to_f32(msA), fbA = bf16_bits_to_f32(mbA);
                    const float fsB = bf16_bits_to_f32(msB), fbB = bf16_bits_to_f32(mbB);
                    advance(meta);
                    load_meta(meta);
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * slot, parity));
                    if (!ok) break;
                    const int g = gc0 + t * kSlices + j;
                    if (g < gc1) {
                        const int gl = g - g_lo;
                        float2 acc[2][V];
                        group_dot<BITS, GS, V>(smem + L.ring + warp * kRingBytesPerWarp + slot * kStageBytes, j, rA,
                                               rB, xs + gl * kXS, p.gsm * kXS, acc);
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            const float sx = sxs[v * p.gsm + gl];
#if defined(QMV_TEST_MUTATE_ORDER)
                            // Test-only build: the streamed kernel folds bias before scale,
                            // so the bit-identity tests can show they detect an order change.
                            if constexpr (V > 1) {
                                part[0][v] = __fmaf_rn(fbA, sx, part[0][v]);
                                part[0][v] = __fmaf_rn(fsA, __fadd_rn(acc[0][v].x, acc[0][v].y), part[0][v]);
                                part[1][v] = __fmaf_rn(fbB, sx, part[1][v]);
                                part[1][v] = __fmaf_rn(fsB, __fadd_rn(acc[1][v].x, acc[1][v].y), part[1][v]);
                                continue;
                            }
#endif
                            part[0][v] = __fmaf_rn(fsA, __fadd_rn(acc[0][v].x, acc[0][v].y), part[0][v]);
                            part[0][v] = __fmaf_rn(fbA, sx, part[0][v]);
                            part[1][v] = __fmaf_rn(fsB, __fadd_rn(acc[1][v].x, acc[1][v].y), part[1][v]);
                            part[1][v] = __fmaf_rn(fbB, sx, part[1][v]);
                        }
                    }
                    __syncwarp();
                    ++consumed;
                    if (lane == 0 && valid(prod)) {
                        fence_proxy_async_smem();
                        issue(prod, issued % kStages);
                        ++issued;
                        advance(prod);
                    }
                }
                if (!ok) break;
                // Step 3: butterfly over the slices; step 4: left fold over chunks.
#pragma unroll
                for (int v = 0; v < V; ++v)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        float t = part[r][v];
                        t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 4));
                        t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 2));
                        t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 1));
                        yr[r][v] = c == 0 ? t : __fadd_rn(yr[r][v], t);
                    }
            }
        }

        if (p.cps == p.ks) {
            if (active && ok) {
#pragma unroll
                for (int v = 0; v < V; ++v)
                    if ((v & 7) == j) {
                        if (nA < p.N) store_y(v, nA, yr[0][v]);
                        if (nB < p.N) store_y(v, nB, yr[1][v]);
                    }
            }
            continue;
        }

        // One chunk per CTA: publish it; the CTA that completes the row tile
        // last folds the chunk values left to right and zeroes what it read,
        // so (with the self-resetting counter) the workspace is zero again.
        if (active && ok) {
#pragma unroll
            for (int v = 0; v < V; ++v)
                if ((v & 7) == j) {
                    float *pp = p.partials + (size_t(chunk_lo) * V + v) * p.N;
                    if (nA < p.N) __stcg(pp + nA, yr[0][v]);
                    if (nB < p.N) __stcg(pp + nB, yr[1][v]);
                }
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_ticket = atomicInc(p.counters + tile, unsigned(p.ks - 1));
        __syncthreads();
        if (s_ticket == unsigned(p.ks - 1)) {
            __threadfence();
            for (int idx = tid; idx < kRowsPerCta * V; idx += kThreads) {
                const int r = idx % kRowsPerCta, v = idx / kRowsPerCta;
                const int n = tile * kRowsPerCta + r;
                if (n >= p.N) continue;
                float *pp = p.partials + size_t(v) * p.N + n;
                float acc = __ldcg(pp);
                __stcg(pp, 0.0f);
                for (int s = 1; s < p.ks; ++s) {
                    float *ps = pp + size_t(s) * V * p.N;
                    acc = __fadd_rn(acc, __ldcg(ps));
                    __stcg(ps, 0.0f);
                }
                store_y(v, n, acc);
            }
        }
        __syncthreads();  // s_ticket is rewritten for the next tile
    }

    if (!ok) {
        // Record the failure, then wait (bounded) for this warp's own copies
        // still in flight before the CTA exits.
        if (lane == 0) atomicOr(p.err, 1u);
        for (int s2 = consumed; s2 < issued; ++s2)
            (void)mbar_wait_bounded(bar0 + 8 * (s2 % kStages), (s2 / kStages) & 1);
    }
}

template <int BITS, int GS>
__global__ void __launch_bounds__(kThreads, 2) qmv_m1(const __grid_constant__ CUtensorMap tmap_w, const Params p)
{
    qmv_body<BITS, GS, 1>(&tmap_w, p);
}

template <int BITS, int GS, int V>
__global__ void __launch_bounds__(kThreads, (V <= 4 ? 2 : 1))
    qmv_streamed(const __grid_constant__ CUtensorMap tmap_w, const Params p)
{
    qmv_body<BITS, GS, V>(&tmap_w, p);
}

}  // namespace qmv
