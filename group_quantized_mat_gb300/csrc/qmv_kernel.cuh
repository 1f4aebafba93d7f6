// sm_103a kernels of the affine group-quantized mat-vec:
//
//   y[m, n] = sum_g ( s[n,g] * sum_{i in g} q[n,i] x[m,i] + b[n,g] * sum_{i in g} x[m,i] )
//
// the factored group dot of mlxcel issue #1289 ("Correction to the obvious
// sketch": scale * accum + sum * bias, no dequantized weight) applied once per
// group (mlxcel PR #1681, "Not covered"), and its order-preserving streamed
// form (#1289 "Step 2"): the weights are read and decoded once and reused for
// V <= 16 activation vectors, each vector's fp32 operation sequence being
// exactly the one an M = 1 launch performs.
//
// Work decomposition (none of it changes the arithmetic):
//  * a row block is 4R consecutive rows; in the warp processing it, lane
//    (p, j), p = lane/8, j = lane%8, owns rows {p, p+4, ..., p+4(R-1)} and
//    slice j of every stage;
//  * a stage is 8 consecutive groups of the row block, one per slice, brought
//    into a private ring of the warp by 2-D TMA boxes (128 bytes x 4R rows,
//    128B-swizzled), one mbarrier per ring slot; lane 0 refills a slot once the
//    warp has read it;
//  * a CTA owns row blocks and a range of K-chunks (see Params); x of its chunk
//    range is staged once into shared memory as fp32, each value
//    pre-multiplied by 2^(-bits * k) (k = its field position inside a 16-bit
//    half word) and padded by 16 bytes per group, so the eight slices hit eight
//    different bank groups; sum(x) per group is staged beside it.
//
// Fixed fp32 order of output (m, n), for every M:
//  1. group: two running sums over even and odd elements, each in increasing
//     order from +0 (one packed fma.rn.f32x2 per element pair): d = a_e + a_o.
//     Every product q*x is exact in fp32 (small integer times 8-bit mantissa);
//  2. fold: P = fma(s_g, d, P); P = fma(b_g, sx_g, P), sx_g = eight sums of
//     eight consecutive x (each left to right) added left to right; P of
//     slice j runs over groups j, j+8, ... of the chunk in increasing order;
//  3. chunk value = butterfly over the eight slices (xor 4, 2, 1);
//  4. y = ((c_0 + c_1) + c_2) + ... over the chunks of kChunkElems elements;
//  5. one rounding to bf16, nearest even.
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

// One wait attempt: the thread may sleep in the instruction (up to the
// suspend-time hint, in ns) until the phase completes.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(1000000u)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: gives up after ~2 s of wall time or 2^24 attempts, whichever
// comes first, so a lost transfer can never hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1; it < (1u << 24); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > 2000000000ull) return false;
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

// Pairs of fp32 values travel as one 64-bit register (low half = first
// element), the operand form of the packed f32x2 instructions.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ float pair_lo(uint64_t v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float pair_hi(uint64_t v) { return __uint_as_float(uint32_t(v >> 32)); }

// Elements of a packed word at masks MASK_LO and MASK_HI, as the exact pair
// (q_lo * 2^(bits*k_lo), q_hi * 2^(bits*k_hi)): each field is OR-ed into the
// significand of 2^23 (one LOP3 each, the mask as immediate, the magic
// constant in a register) and 2^23 is subtracted from both halves at once.
template <uint32_t MASK_LO, uint32_t MASK_HI>
__device__ __forceinline__ uint64_t field_pair(uint32_t w, uint32_t magic, uint64_t neg_magic2)
{
    uint64_t d;
    asm("{\n\t.reg .b32 lo, hi;\n\t.reg .b64 t;\n\t"
        "lop3.b32 lo, %1, %2, %4, 0xEA;\n\t"
        "lop3.b32 hi, %1, %3, %4, 0xEA;\n\t"
        "mov.b64 t, {lo, hi};\n\t"
        "add.rn.f32x2 %0, t, %5;\n\t}"
        : "=l"(d)
        : "r"(w), "n"(MASK_LO), "n"(MASK_HI), "r"(magic), "l"(neg_magic2));
    return d;
}

// Element pairs (2p, 2p+1) of one packed word, as exact floats q * 2^(bits*k),
// k the element's position inside its 16-bit half. The matching x values were
// staged pre-multiplied by 2^(-bits*k), so each product equals q * x exactly.
template <int BITS>
__device__ __forceinline__ void extract_pairs(uint32_t w, uint32_t magic, uint64_t nm, uint64_t (&q)[16 / BITS])
{
    // w >> 16 as a multiply-high, which runs on the FMA pipe (the extraction
    // keeps the integer/logic pipe busy).
    uint32_t hi;
    asm("mul.hi.u32 %0, %1, 65536;" : "=r"(hi) : "r"(w));
    const uint32_t lo = w;
    if constexpr (BITS == 4) {
        q[0] = field_pair<0x000Fu, 0x00F0u>(lo, magic, nm);
        q[1] = field_pair<0x0F00u, 0xF000u>(lo, magic, nm);
        q[2] = field_pair<0x000Fu, 0x00F0u>(hi, magic, nm);
        q[3] = field_pair<0x0F00u, 0xF000u>(hi, magic, nm);
    } else {
        q[0] = field_pair<0x0003u, 0x000Cu>(lo, magic, nm);
        q[1] = field_pair<0x0030u, 0x00C0u>(lo, magic, nm);
        q[2] = field_pair<0x0300u, 0x0C00u>(lo, magic, nm);
        q[3] = field_pair<0x3000u, 0xC000u>(lo, magic, nm);
        q[4] = field_pair<0x0003u, 0x000Cu>(hi, magic, nm);
        q[5] = field_pair<0x0030u, 0x00C0u>(hi, magic, nm);
        q[6] = field_pair<0x0300u, 0x0C00u>(hi, magic, nm);
        q[7] = field_pair<0x3000u, 0xC000u>(hi, magic, nm);
    }
}

__device__ __forceinline__ void lds_v2_u64(uint32_t addr, uint64_t &a, uint64_t &b)
{
    asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
}

__device__ __forceinline__ uint4 lds_v4_u32(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &c, int k)
{
    return k == 0 ? c.x : (k == 1 ? c.y : (k == 2 ? c.z : c.w));
}

// ----------------------------------------------------------- group dot --

// Step 1 of the fixed order for one group of the lane's R rows against V
// staged vectors: acc[r][v] = (a_e, a_o) as one 64-bit pair.
//   box     shared address of the stage;
//   woff[r] byte offset in the stage of the first 16-byte chunk of slice j's
//           group in row pr + 4r (128B swizzle applied; chunk c of the group
//           sits at woff ^ (c << 4));
//   xg      shared address of the group's staged x (vector 0); xvstride in bytes.
template <int BITS, int GS, int V, int R>
__device__ __forceinline__ void group_dot(uint32_t box, const uint32_t (&woff)[R], uint32_t xg, uint32_t xvstride,
                                          uint32_t magic, uint64_t nm, uint64_t (&acc)[R][V])
{
    constexpr int kChunks = group_bytes(BITS, GS) / 16;
    constexpr int kPerWord = 32 / BITS;

    uint4 w[R][kChunks];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < kChunks; ++c) w[r][c] = lds_v4_u32(box + (woff[r] ^ (c << 4)));
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < V; ++v) acc[r][v] = 0ull;
#pragma unroll
    for (int wi = 0; wi < kChunks * 4; ++wi) {
        uint64_t q[R][kPerWord / 2];
#pragma unroll
        for (int r = 0; r < R; ++r) extract_pairs<BITS>(word_of(w[r][wi / 4], wi % 4), magic, nm, q[r]);
#pragma unroll
        for (int v = 0; v < V; ++v) {
#pragma unroll
            for (int hh = 0; hh < kPerWord / 4; ++hh) {
                uint64_t x01, x23;
                lds_v2_u64(xg + v * xvstride + (wi * kPerWord + hh * 4) * 4, x01, x23);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    acc[r][v] = ffma2(q[r][2 * hh], x01, acc[r][v]);
                    acc[r][v] = ffma2(q[r][2 * hh + 1], x23, acc[r][v]);
                }
            }
        }
    }
}

// ---------------------------------------------------------------- kernel --

template <int BITS, int GS, int V, int R>
__device__ __forceinline__ void qmv_body(const CUtensorMap *tmap_w, const Params &p)
{
    constexpr int RW = 4 * R;  // rows per row block (one warp's rows)
    constexpr int kGB = group_bytes(BITS, GS);
    constexpr int kGPB = groups_per_box(BITS, GS);
    constexpr int kBPS = boxes_per_stage(BITS, GS);
    constexpr int kCG = chunk_groups(GS);
    constexpr int kSPC = kCG / kSlices;  // stages per full chunk (4 or 2)
    constexpr int kXS = x_stride(GS);
    constexpr int kPerHalf = 16 / BITS;
    constexpr int kBoxSmem = kBoxBytes * RW;
    constexpr int kStageBytes = kBPS * kBoxSmem;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ unsigned s_ticket;
    // Align the dynamic base to 1024 bytes (the 128B swizzle pattern repeats
    // every 1024 bytes) by offsetting the __shared__ array itself, so every
    // access below stays a shared-memory access.
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int nwarps = p.warps;
    const int nthreads = nwarps * 32;
    const int tile_rows = p.RB * RW;  // rows the CTA's chunk-value buffer holds
    const SmemLayout L = smem_layout(BITS, GS, V, RW, nwarps, p.stages, p.gsm, p.cps, tile_rows);
    float *xs = reinterpret_cast<float *>(smem + L.xs);
    float *sxs = reinterpret_cast<float *>(smem + L.sx);
    float *cvs = reinterpret_cast<float *>(smem + L.cv);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pr = lane >> 3, j = lane & 7;
    const int c_lo = blockIdx.y * p.cps;
    const int c_hi = c_lo + p.cps < p.ks ? c_lo + p.cps : p.ks;
    const int ncta = c_hi - c_lo;
    const int g_lo = c_lo * kCG;
    const int g_hi = c_hi * kCG < p.G ? c_hi * kCG : p.G;
    const int gsn = g_hi - g_lo;  // groups of x staged by this CTA
    // Row blocks of this CTA: a balanced share of all NB row blocks (persistent
    // grid), or RB consecutive ones (one row tile per CTA).
    int rb_lo, rb_hi;
    if (p.balanced) {
        rb_lo = int((long long)blockIdx.x * p.NB / gridDim.x);
        rb_hi = int((long long)(blockIdx.x + 1) * p.NB / gridDim.x);
    } else {
        rb_lo = blockIdx.x * p.RB;
        rb_hi = rb_lo + p.RB < p.NB ? rb_lo + p.RB : p.NB;
    }
    const int row_t0 = rb_lo * RW;
    const int nunits = (rb_hi - rb_lo) * p.H;  // (row block, chunk phase) pairs
    const int stage_shift = __ffs(p.stages) - 1;

    // A unit is one row block and the contiguous chunk block [cb0, cb1) of its
    // chunk phase: groups [gw0, gw1), stage s holding groups gw0 + 8s .. + 7; a
    // chunk ends every kSPC stages and only the unit's last stage can be partial.
    struct Unit {
        int row0, cb0, gw0, gw1, total;
    };
    auto unit_geo = [&](int u) {
        Unit q;
        const int rbl = u / p.H, hh = u - rbl * p.H;
        q.row0 = (rb_lo + rbl) * RW;
        q.cb0 = c_lo + hh * ncta / p.H;
        const int cb1 = c_lo + (hh + 1) * ncta / p.H;
        q.gw0 = q.cb0 * kCG;
        q.gw1 = cb1 * kCG < p.G ? cb1 * kCG : p.G;
        q.total = (q.gw1 - q.gw0 + kSlices - 1) / kSlices;
        return q;
    };

    const uint32_t bar0 = smem_u32(bars + warp * p.stages);
    const uint32_t ring_w = smem_u32(smem + L.ring + warp * p.stages * kStageBytes);
    const uint64_t pol = l2_evict_first_policy();

    // Producer (lane 0): the warp's stage sequence runs through its units
    // u = warp, warp + nwarps, ... in order; `issued` counts stages issued.
    int pu = warp, ps = 0, issued = 0;
    Unit pg = unit_geo(pu < nunits ? pu : 0);
    auto issue_next = [&]() {
        if (pu >= nunits) return;
        const int slot = issued & (p.stages - 1);
        const int gst = pg.gw0 + ps * kSlices;  // first group of the stage
        int nb = (pg.gw1 - gst + kGPB - 1) / kGPB;
        nb = nb < kBPS ? nb : kBPS;
        mbar_arrive_expect_tx(bar0 + 8 * slot, nb * kBoxSmem);
        for (int b = 0; b < nb; ++b)
            tma_load_2d(ring_w + slot * kStageBytes + b * kBoxSmem, tmap_w, gst * kGB + b * kBoxBytes, pg.row0,
                        bar0 + 8 * slot, pol);
        ++issued;
        if (++ps == pg.total) {
            ps = 0;
            pu += nwarps;
            if (pu < nunits) pg = unit_geo(pu);
        }
    };

    // Weight tiles first: they do not depend on x, so their latency overlaps the staging below.
    if (lane == 0) {
        for (int s = 0; s < p.stages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
        for (int s = 0; s < p.stages; ++s) issue_next();
    }
    __syncwarp();

    // Stage x for groups [g_lo, g_hi): fp32, position-scaled, 8 elements per task.
    {
        constexpr int kUPG = GS / 8;
        const int per_vec = gsn * kUPG, all = V * per_vec;
        for (int u0 = tid; u0 < all; u0 += 4 * nthreads) {
            uint4 raw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int u = u0 + k * nthreads;
                if (u < all) {
                    const int v = u / per_vec, rem = u - v * per_vec;
                    raw[k] = __ldg(reinterpret_cast<const uint4 *>(p.x + size_t(v) * p.K + size_t(g_lo) * GS) + rem);
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int u = u0 + k * nthreads;
                if (u < all) {
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
        // each left to right, then those (eight, or sixteen for gs = 128) left to right.
        for (int idx = tid; idx < V * gsn; idx += nthreads) {
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

    bool ok = true;
    int consumed = 0;
    // The magic constant and the pair (-2^23, -2^23) as register operands of the extraction.
    uint32_t magic;
    asm volatile("mov.b32 %0, %1;" : "=r"(magic) : "n"(kMagic));
    const uint64_t nm = 0xCB000000CB000000ull;
    // Per-lane byte offsets, inside a stage, of the first chunk of slice j's
    // group for each of the lane's rows (128B swizzle: chunk index XOR row % 8).
    uint32_t woff[R];
    {
        constexpr int kChunks = kGB / 16;
        const int c0 = (j % kGPB) * kChunks;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = pr + 4 * r;
            woff[r] = uint32_t((j / kGPB) * kBoxSmem + row * kBoxBytes + ((c0 ^ (row & 7)) << 4));
        }
    }
    const uint32_t ring_s = smem_u32(smem + L.ring);
    const uint32_t xs_s = smem_u32(xs);

    for (int u = warp; u < nunits && ok; u += nwarps) {
        const Unit q = unit_geo(u);
        const int rbl = u / p.H;
        // Scale and bias of the lane's group, loaded one stage ahead.
        const uint16_t *srow[R], *brow[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int n = q.row0 + pr + 4 * r < p.N ? q.row0 + pr + 4 * r : p.N - 1;
            srow[r] = p.scales + size_t(n) * p.G;
            brow[r] = p.biases + size_t(n) * p.G;
        }
        uint16_t ms[R], mb[R];
        {
            const int g = q.gw0 + j < q.gw1 ? q.gw0 + j : q.gw1 - 1;
#pragma unroll
            for (int r = 0; r < R; ++r) { ms[r] = __ldg(srow[r] + g); mb[r] = __ldg(brow[r] + g); }
        }
        float part[R][V];
        for (int s = 0; s < q.total; ++s) {
            const int t = s & (kSPC - 1);
            if (t == 0) {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int v = 0; v < V; ++v) part[r][v] = 0.0f;
            }
            float fs[R], fb[R];
#pragma unroll
            for (int r = 0; r < R; ++r) { fs[r] = bf16_bits_to_f32(ms[r]); fb[r] = bf16_bits_to_f32(mb[r]); }
            const int g = q.gw0 + s * kSlices + j;
            if (s + 1 < q.total) {
                const int gn = g + kSlices < q.gw1 ? g + kSlices : q.gw1 - 1;
#pragma unroll
                for (int r = 0; r < R; ++r) { ms[r] = __ldg(srow[r] + gn); mb[r] = __ldg(brow[r] + gn); }
            }
            const int slot = consumed & (p.stages - 1);
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * slot, (consumed >> stage_shift) & 1));
            if (!ok) break;
            if (g < q.gw1) {
                const int gl = g - g_lo;
                uint64_t acc[R][V];
                group_dot<BITS, GS, V, R>(ring_s + (warp * p.stages + slot) * kStageBytes, woff,
                                          xs_s + gl * kXS * 4, p.gsm * kXS * 4, magic, nm, acc);
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const float sx = sxs[v * p.gsm + gl];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float d = __fadd_rn(pair_lo(acc[r][v]), pair_hi(acc[r][v]));
#if defined(QMV_TEST_MUTATE_ORDER)
                        // Test-only build: the streamed kernel folds bias before scale,
                        // so the bit-identity tests can show they detect an order change.
                        if constexpr (V > 1) {
                            part[r][v] = __fmaf_rn(fb[r], sx, part[r][v]);
                            part[r][v] = __fmaf_rn(fs[r], d, part[r][v]);
                            continue;
                        }
#endif
                        part[r][v] = __fmaf_rn(fs[r], d, part[r][v]);
                        part[r][v] = __fmaf_rn(fb[r], sx, part[r][v]);
                    }
                }
            }
            __syncwarp();
            ++consumed;
            if (lane == 0) {
                fence_proxy_async_smem();
                issue_next();
            }
            // End of a chunk: butterfly over the slices, chunk value to shared memory.
            if (t == kSPC - 1 || s == q.total - 1) {
                float *cv = cvs + ((q.cb0 + s / kSPC - c_lo) * tile_rows + rbl * RW) * V;
#pragma unroll
                for (int v = 0; v < V; ++v)
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        float x1 = part[r][v];
                        x1 = __fadd_rn(x1, __shfl_xor_sync(0xffffffffu, x1, 4));
                        x1 = __fadd_rn(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
                        x1 = __fadd_rn(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
                        if ((v & 7) == j) cv[(pr + 4 * r) * V + v] = x1;
                    }
            }
        }
    }
    if (!ok && lane == 0) {
        // Record the failure, then wait (bounded) for this warp's own copies
        // still in flight before the CTA may exit.
        atomicOr(p.err, 1u);
        for (int s2 = consumed; s2 < issued; ++s2)
            (void)mbar_wait_bounded(bar0 + 8 * (s2 & (p.stages - 1)), (s2 >> stage_shift) & 1);
    }
    __syncthreads();

    auto store_y = [&](int v, int n, float val) {
        if (p.f32_out)
            static_cast<float *>(p.y)[size_t(v) * p.N + n] = val;
        else
            static_cast<__nv_bfloat16 *>(p.y)[size_t(v) * p.N + n] = __float2bfloat16_rn(val);
    };
    const int nrows = (rb_hi - rb_lo) * RW;

    // Step 4: fold the chunk values left to right.
    if (p.cps == p.ks) {
        for (int idx = tid; idx < nrows * V; idx += nthreads) {
            const int r = idx / V, v = idx - r * V;
            const int n = row_t0 + r;
            if (n >= p.N) continue;
            float acc = cvs[r * V + v];
            for (int c = 1; c < p.ks; ++c) acc = __fadd_rn(acc, cvs[(c * tile_rows + r) * V + v]);
            store_y(v, n, acc);
        }
        return;
    }

    // One chunk per CTA: publish its values; the CTA that completes the row
    // tile last folds all chunks left to right and zeroes what it read, so
    // (with the self-resetting counter) the workspace is zero again.
    for (int idx = tid; idx < nrows * V; idx += nthreads) {
        const int r = idx / V, v = idx - r * V;
        const int n = row_t0 + r;
        if (n < p.N) __stcg(p.partials + (size_t(c_lo) * V + v) * p.N + n, cvs[r * V + v]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_ticket = atomicInc(p.counters + blockIdx.x, unsigned(p.ks - 1));
    __syncthreads();
    if (s_ticket != unsigned(p.ks - 1)) return;
    __threadfence();
    for (int idx = tid; idx < nrows * V; idx += nthreads) {
        const int r = idx % nrows, v = idx / nrows;
        const int n = row_t0 + r;
        if (n >= p.N) continue;
        float *pp = p.partials + size_t(v) * p.N + n;
        float acc = __ldcg(pp);
        __stcg(pp, 0.0f);
        for (int c = 1; c < p.ks; ++c) {
            float *pc = pp + size_t(c) * V * p.N;
            acc = __fadd_rn(acc, __ldcg(pc));
            __stcg(pc, 0.0f);
        }
        store_y(v, n, acc);
    }
}

// Rows per lane R: the single-vector kernel comes with R = 2 and R = 4 (the
// host picks by shape); the streamed kernel uses R = 2 (its registers go to V).
template <int BITS, int GS, int R>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) qmv_m1(const __grid_constant__ CUtensorMap tmap_w, const Params p)
{
    qmv_body<BITS, GS, 1, R>(&tmap_w, p);
}

template <int BITS, int GS, int V>
__global__ void __launch_bounds__(kMaxWarps * 16, (V <= 4 ? 2 : 1))
    qmv_streamed(const __grid_constant__ CUtensorMap tmap_w, const Params p)
{
    qmv_body<BITS, GS, V, 2>(&tmap_w, p);
}

}  // namespace qmv
