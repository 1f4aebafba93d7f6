// sm_103a kernel of the affine group-quantized mat-vec:
//
//   y[m, n] = sum_g ( s[n,g] * sum_{i in g} q[n,i] x[m,i] + b[n,g] * sum_{i in g} x[m,i] )
//
// evaluated in the factored form of mlxcel issue #1289 ("Correction to the
// obvious sketch": scale * accum + sum * bias, no dequantized weight) and
// streamed for V <= 16 activation vectors from one read of the weights
// (#1289 "Step 2"), each vector's fp32 operation sequence being exactly the one
// a V = 1 launch performs.
//
// Fixed fp32 order of output (m, n), the same for every V:
//  1. subgroup t (64 consecutive elements of row n, inside one quantization
//     group g): with E the largest exponent field among its 64 bf16 x values
//     (at least 1), every product is q_i * x_i * 2^(105 - E), formed exactly
//     inside an fma. Two running sums a_e, a_o over the even and odd elements
//     in processing order from +0, one fma per element;
//     d = ((a_e + a_o) * f1) * f2 with f1 * f2 = 2^(E - 105).
//     The kernels reach the same product two ways (below, "field readings");
//     an x_i whose exponent field is more than 231 below E is staged as a
//     zero of its sign in both (its product would lie below 2^-247, far under
//     the fp32 grid), so that both stagings are exact for every other x_i;
//  2. term = fma(s_g, d, b_g * sx), sx = sum of the subgroup's 64 x: eight
//     sums of eight consecutive elements (each left to right) added left to
//     right;
//  3. chunk value (32 subgroups, 2048 elements; lanes past the row's end add
//     +0) = binary tree over the 32 subgroup slots l: pairs (l, l^16) first,
//     then (l, l^8), (l, l^4), (l, l^2), (l, l^1);
//  4. y = ((c_0 + c_1) + c_2) + ... over the chunks of the row;
//  5. one rounding to bf16, nearest even.
// Field readings (both give the products of step 1 bit for bit):
//  * qmv_streamed: x'_i = x_i * 2^(254 - bits*k_i - E), k_i = position of
//    element i inside its 16-bit half word, exactly a bf16 value, staged as
//    fp32; field q_i is the fp32 whose bit pattern is q_i << (bits*k_i), the
//    subnormal q_i * 2^(bits*k_i - 149); one fma.rn.f32x2 per element pair.
//  * qmv_m1: x''_i = x_i * 2^(238 - bits*j_i - E), j_i = position of the
//    field inside its byte, staged as bf16; field q_i is the bf16 half whose
//    bit pattern is q_i << (bits*j_i), i.e. q_i * 2^(bits*j_i - 133) (the low
//    byte of a bf16 read as an integer n is n * 2^-133 exactly). One mask
//    isolates two fields (one per 16-bit half), and fma.rn.f32.bf16 (exact
//    product, fp32 sum, one rounding) takes each half: half the integer work
//    of the fp32 reading, which is what bounds a one-vector pass.
// Processing order inside a 4-bit subgroup: its two 16-byte halves, the half
// selected by bit 2 of the subgroup index first (that keeps the eight lanes of
// a shared-memory phase on distinct banks when a warp reads 32 subgroups of a
// row); inside a half, increasing element order. 2-bit subgroups run in
// increasing element order.
//
// Work decomposition (none of it changes the arithmetic): a unit is 4 rows x
// some chunks; lane l of the warp processing a unit owns subgroup l of each
// of its chunks in all 4 rows. Warps take units from a shared counter.
//  * qmv_m1 (one vector): producer warps stream units (4 whole rows in one
//    1-D bulk copy when they fit, else 4 rows x some chunks as one 2-D
//    tensor-map tile or one copy per row, plus tensor-map boxes of the rows'
//    scales and biases) into a CTA-wide ring of shared-memory slots, one
//    "full" and one "empty" mbarrier per slot; consumer warps compute them.
//    The CTA's x arrives by one bulk copy and is staged in place.
//  * qmv_streamed (V vectors): qmv_stage_x stages every vector's x' once per
//    call into the workspace; the CTA brings in its range with one bulk copy
//    per vector. A warp loads its unit's bytes (the lane's own subgroup of 4
//    rows of one chunk), scales and biases straight into registers; V times
//    the arithmetic hides the latency.
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

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// One wait attempt: the thread may wait in the instruction for a
// system-dependent time before it reports the phase still open. (No
// suspend-time hint: with one, waiting warps measured up to 1 % slower to
// resume.)
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

// 1-D bulk copy global -> this CTA's shared memory (16-byte aligned addresses,
// size a multiple of 16), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// The same without an L2 hint.
__device__ __forceinline__ void bulk_load_plain(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// 1-D tensor-map box load at element coordinate x (a multiple of 8 for
// 2-byte elements); elements past the tensor's end arrive as zeros.
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const CUtensorMap *map, int x, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2}], [%3];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(bar)
        : "memory");
}

// 2-D tensor-map box load at element coordinates (x, y), x * element size a
// multiple of 16 bytes; elements outside the tensor arrive as zeros.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Programmatic dependent launch: wait until the preceding grid on the stream
// has completed and its memory is visible (returns at once when the launch had
// no programmatic dependency), and allow the next grid to be scheduled.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

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

__device__ __forceinline__ void sts_v4_u32(uint32_t addr, const uint4 &v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// ------------------------------------------------------- the datapath --

// Pairs of fp32 values travel as one 64-bit register (low half = first
// element), the operand form of the packed f32x2 instructions.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}

__device__ __forceinline__ float pair_lo(uint64_t v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float pair_hi(uint64_t v) { return __uint_as_float(uint32_t(v >> 32)); }

// w >> 16 as a multiply-high, which runs on the FMA pipe (the field masks keep
// the integer/logic pipe busy).
__device__ __forceinline__ uint32_t hi_half(uint32_t w)
{
    uint32_t h;
    asm("mul.hi.u32 %0, %1, 65536;" : "=r"(h) : "r"(w));
    return h;
}

// a + (bf16 half WH of w) * (bf16 half XH of x): exact product, fp32 sum,
// one rounding.
template <int WH, int XH>
__device__ __forceinline__ float fma_bf16(uint32_t w, uint32_t x, float a)
{
    float d;
    if constexpr (WH == 0 && XH == 0)
        asm("{.reg .b16 wl, wh, xl, xh;\n\tmov.b32 {wl, wh}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, wl, xl, %3;}" : "=f"(d) : "r"(w), "r"(x), "f"(a));
    else if constexpr (WH == 0)
        asm("{.reg .b16 wl, wh, xl, xh;\n\tmov.b32 {wl, wh}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, wl, xh, %3;}" : "=f"(d) : "r"(w), "r"(x), "f"(a));
    else if constexpr (XH == 0)
        asm("{.reg .b16 wl, wh, xl, xh;\n\tmov.b32 {wl, wh}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, wh, xl, %3;}" : "=f"(d) : "r"(w), "r"(x), "f"(a));
    else
        asm("{.reg .b16 wl, wh, xl, xh;\n\tmov.b32 {wl, wh}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, wh, xh, %3;}" : "=f"(d) : "r"(w), "r"(x), "f"(a));
    return d;
}

// The four element pairs of an octet (8 consecutive elements in processing
// order) as fp32 bit patterns q << (bits*k): one mask per element.
//   4-bit: the octet is one word; pairs (0,1), (2,3) from its low half and
//          (4,5), (6,7) from its high half `h`.
//   2-bit: the octet is one 16-bit half `u` of a word.
__device__ __forceinline__ void octet_pairs4(uint32_t w, uint32_t h, uint64_t (&q)[4])
{
    q[0] = pack2(w & 0x000Fu, w & 0x00F0u);
    q[1] = pack2(w & 0x0F00u, w & 0xF000u);
    q[2] = pack2(h & 0x000Fu, h & 0x00F0u);
    q[3] = pack2(h & 0x0F00u, h & 0xF000u);
}

__device__ __forceinline__ void octet_pairs2(uint32_t u, uint64_t (&q)[4])
{
    q[0] = pack2(u & 0x0003u, u & 0x000Cu);
    q[1] = pack2(u & 0x0030u, u & 0x00C0u);
    q[2] = pack2(u & 0x0300u, u & 0x0C00u);
    q[3] = pack2(u & 0x3000u, u & 0xC000u);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &c, int k)
{
    return k == 0 ? c.x : (k == 1 ? c.y : (k == 2 ? c.z : c.w));
}

// Pairs of octet `o` (0..7 in processing order) of a subgroup, for BITS.
// quads[p] = the subgroup's 16-byte pieces in processing order (4-bit: two
// pieces; 2-bit: one).
template <int BITS>
__device__ __forceinline__ void subgroup_octet(const uint4 (&quads)[BITS == 4 ? 2 : 1], int o, uint64_t (&q)[4])
{
    if constexpr (BITS == 4) {
        const uint32_t w = word_of(quads[o >> 2], o & 3);
        octet_pairs4(w, hi_half(w), q);
    } else {
        const uint32_t w = word_of(quads[0], o >> 1);
        octet_pairs2((o & 1) ? hi_half(w) : w, q);
    }
}

// Byte offsets, inside a row's copy of a chunk, of the lane's subgroup pieces
// in processing order (4-bit: the half selected by bit 2 of the lane first).
template <int BITS>
__device__ __forceinline__ void piece_offsets(int lane, uint32_t (&off)[BITS == 4 ? 2 : 1])
{
    if constexpr (BITS == 4) {
        const uint32_t first = ((lane >> 2) & 1) * 16u;
        off[0] = uint32_t(lane) * 32u + first;
        off[1] = uint32_t(lane) * 32u + (16u - first);
    } else {
        off[0] = uint32_t(lane) * 16u;
    }
}

// Step 1 for V = 1 in the bf16 field reading: ae[r], ao[r] of the lane's
// subgroup in rows 0..3.
//   quads[r]  the subgroup's bytes in row r (16-byte pieces, processing order);
//   xsub      shared address of the staged subgroup (64 bf16 x'', octet o in
//             processing order at 16 * (o ^ sw)).
// A 4-bit octet is one word w: fields (0,4), (1,5), (2,6), (3,7) sit in the
// two halves of w & 0x000F000F, w & 0x00F000F0 and the same masks of w >> 8.
// A 2-bit word holds octets 2p (low halves) and 2p + 1 (high halves): fields
// k and k + 4 of both in the masks 3 << 2k of w and of w >> 8.
//   SWZ       false: octet o at xsub + 16 * o instead (no swizzle).
template <int BITS, bool SWZ = true>
__device__ __forceinline__ void subgroup_dot_v1(const uint4 (&quads)[kRows][BITS == 4 ? 2 : 1], uint32_t xsub, uint32_t sw,
                                                float (&ae)[kRows], float (&ao)[kRows])
{
    auto oct = [&](int o) { return SWZ ? xsub + ((uint32_t(o) ^ sw) << 4) : xsub + (uint32_t(o) << 4); };
#pragma unroll
    for (int r = 0; r < kRows; ++r) ae[r] = ao[r] = 0.0f;
    if constexpr (BITS == 4) {
#pragma unroll
        for (int o = 0; o < 8; ++o) {
            const uint4 X = lds_v4_u32(oct(o));
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const uint32_t w = word_of(quads[r][o >> 2], o & 3), w8 = w >> 8;
                const uint32_t m0 = w & 0x000F000Fu, m1 = w & 0x00F000F0u;
                const uint32_t m2 = w8 & 0x000F000Fu, m3 = w8 & 0x00F000F0u;
                ae[r] = fma_bf16<0, 0>(m0, X.x, ae[r]);
                ao[r] = fma_bf16<0, 1>(m1, X.x, ao[r]);
                ae[r] = fma_bf16<0, 0>(m2, X.y, ae[r]);
                ao[r] = fma_bf16<0, 1>(m3, X.y, ao[r]);
                ae[r] = fma_bf16<1, 0>(m0, X.z, ae[r]);
                ao[r] = fma_bf16<1, 1>(m1, X.z, ao[r]);
                ae[r] = fma_bf16<1, 0>(m2, X.w, ae[r]);
                ao[r] = fma_bf16<1, 1>(m3, X.w, ao[r]);
            }
        }
    } else {
#pragma unroll
        for (int pw = 0; pw < 4; ++pw) {
            const uint4 X0 = lds_v4_u32(oct(2 * pw));
            const uint4 X1 = lds_v4_u32(oct(2 * pw + 1));
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const uint32_t w = word_of(quads[r][0], pw), w8 = w >> 8;
                uint32_t m[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    m[k] = w & (0x00030003u << (2 * k));
                    m[k + 4] = w8 & (0x00030003u << (2 * k));
                }
                ae[r] = fma_bf16<0, 0>(m[0], X0.x, ae[r]);
                ao[r] = fma_bf16<0, 1>(m[1], X0.x, ao[r]);
                ae[r] = fma_bf16<0, 0>(m[2], X0.y, ae[r]);
                ao[r] = fma_bf16<0, 1>(m[3], X0.y, ao[r]);
                ae[r] = fma_bf16<0, 0>(m[4], X0.z, ae[r]);
                ao[r] = fma_bf16<0, 1>(m[5], X0.z, ao[r]);
                ae[r] = fma_bf16<0, 0>(m[6], X0.w, ae[r]);
                ao[r] = fma_bf16<0, 1>(m[7], X0.w, ao[r]);
                ae[r] = fma_bf16<1, 0>(m[0], X1.x, ae[r]);
                ao[r] = fma_bf16<1, 1>(m[1], X1.x, ao[r]);
                ae[r] = fma_bf16<1, 0>(m[2], X1.y, ae[r]);
                ao[r] = fma_bf16<1, 1>(m[3], X1.y, ao[r]);
                ae[r] = fma_bf16<1, 0>(m[4], X1.z, ae[r]);
                ao[r] = fma_bf16<1, 1>(m[5], X1.z, ao[r]);
                ae[r] = fma_bf16<1, 0>(m[6], X1.w, ae[r]);
                ao[r] = fma_bf16<1, 1>(m[7], X1.w, ao[r]);
            }
        }
    }
}

// Step 1 for VP vectors: acc[r][v].
//   xsub   shared address of vector 0's staged subgroup (fp32 x', octet o at
//          32 * o); xv bytes between vectors.
template <int BITS, int VP>
__device__ __forceinline__ void subgroup_dot_vp(const uint4 (&quads)[kRows][BITS == 4 ? 2 : 1], uint32_t xsub,
                                                uint32_t xv, uint64_t (&acc)[kRows][VP])
{
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int v = 0; v < VP; ++v) acc[r][v] = 0ull;
#pragma unroll
    for (int o = 0; o < 8; ++o) {
        uint64_t q[kRows][4];
#pragma unroll
        for (int r = 0; r < kRows; ++r) subgroup_octet<BITS>(quads[r], o, q[r]);
#pragma unroll
        for (int v = 0; v < VP; ++v) {
            uint64_t x01, x23, x45, x67;
            lds_v2_u64(xsub + v * xv + o * 32, x01, x23);
            lds_v2_u64(xsub + v * xv + o * 32 + 16, x45, x67);
            // pair by pair, the four rows' chains side by side (each chain's
            // own order is unchanged)
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r][v] = ffma2(q[r][0], x01, acc[r][v]);
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r][v] = ffma2(q[r][1], x23, acc[r][v]);
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r][v] = ffma2(q[r][2], x45, acc[r][v]);
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r][v] = ffma2(q[r][3], x67, acc[r][v]);
        }
    }
}

// subgroup_dot_vp with the weight bytes re-read from shared memory (cell
// (r, pc) of this lane at wcell + (r*NP + pc) * 512), for two-pass V.
template <int BITS, int VP>
__device__ __forceinline__ void subgroup_dot_vp_smem(uint32_t wcell, uint32_t xsub, uint32_t xv,
                                                     uint64_t (&acc)[kRows][VP])
{
    constexpr int NP = BITS == 4 ? 2 : 1;
    uint4 quads[kRows][NP];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int pc = 0; pc < NP; ++pc) quads[r][pc] = lds_v4_u32(wcell + uint32_t(r * NP + pc) * 512u);
    subgroup_dot_vp<BITS, VP>(quads, xsub, xv, acc);
}

// Step 2: the subgroup's term from its pair sums.
template <bool STREAMED>
__device__ __forceinline__ float subgroup_term(float ae, float ao, float s, float b, float sx, float f1, float f2)
{
    float d = __fadd_rn(ae, ao);
    d = __fmul_rn(__fmul_rn(d, f1), f2);
#if defined(QMV_TEST_MUTATE_ORDER)
    // Test-only build: the streamed kernel adds the bias term last instead, a
    // different fp32 order that the bit-identity tests must be able to detect.
    if constexpr (STREAMED) return __fadd_rn(__fmul_rn(s, d), __fmul_rn(b, sx));
#endif
    return __fmaf_rn(s, d, __fmul_rn(b, sx));
}

// Step 3 for N values per lane (N a power of two, at most 32): the binary
// tree over the 32 lanes, as a reduce-scatter. At the step with mask m a lane
// keeps half of its values (the upper half if lane & m) and adds its
// partner's copy of them, so every partial sum is exactly the tree's. After
// log2(N) steps lane l holds value index l >> (5 - log2 N); the remaining
// steps are plain butterflies. Returns that value (the full 32-lane sum).
template <int N>
__device__ __forceinline__ float tree_reduce_scatter(float (&val)[N], int lane)
{
    constexpr int LOG = N == 1 ? 0 : N == 2 ? 1 : N == 4 ? 2 : N == 8 ? 3 : N == 16 ? 4 : 5;
    static_assert((1 << LOG) == N, "N must be a power of two <= 32");
#pragma unroll
    for (int step = 0; step < LOG; ++step) {
        const int m = 16 >> step;
        const int half = N >> (step + 1);
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float keep = upper ? val[half + i] : val[i];
            const float send = upper ? val[i] : val[half + i];
            val[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, m));
        }
    }
    float t = val[0];
#pragma unroll
    for (int step = LOG; step < 5; ++step) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, 16 >> step));
    return t;
}

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// ---------------------------------------------------------------- kernel --

template <int BITS, int V>
struct Traits {
    static constexpr int VP = vectors_per_pass(V);
    static constexpr int PASSES = (V + VP - 1) / VP;
    static constexpr int NVAL = kRows * VP;
    static constexpr int NRED = NVAL <= 4 ? 4 : NVAL <= 8 ? 8 : NVAL <= 16 ? 16 : 32;
    static constexpr int NP = BITS == 4 ? 2 : 1;              // 16-byte pieces per subgroup row
    // Two equal passes of at least 7 vectors (V = 14, 16): each pass of a unit
    // is a work item of its own (both load the unit's weights), so a CTA's
    // last items spread over more warps (V = 16: 6 % faster). Otherwise a
    // unit's passes form one item, its weights parked in shared memory
    // between them (splitting them measured 1-6 % slower there).
    static constexpr bool SPLIT = PASSES == 2 && 2 * VP == V && VP >= 7;
    static constexpr int IPU = SPLIT ? PASSES : 1;  // work items per unit
    static constexpr int PPI = SPLIT ? 1 : PASSES;  // passes per work item
};

// Steps 1 and 2 for eight consecutive elements of a subgroup, held as raw
// bf16 by each of eight consecutive lanes (all 32 lanes of the warp call
// this): their staged x' as four bf16 pairs, and the subgroup's
// (sx, f1, f2, 0). BF16_FIELDS selects the scaling of the bf16 field reading
// (x''), else that of the fp32 field reading (x').
template <int BITS, bool BF16_FIELDS>
__device__ __forceinline__ void stage_eight(const uint4 &raw, uint4 &packed, float4 &meta)
{
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t bits[8], e = 1, emin = 255;
    float xv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        bits[i] = (i & 1) ? (w4[i / 2] >> 16) : (w4[i / 2] & 0xFFFFu);
        xv[i] = bf16_bits_to_f32(bits[i]);
        const uint32_t f = (bits[i] >> 7) & 0xFFu;
        e = f > e ? f : e;
        emin = f < emin ? f : emin;
    }
    // largest exponent field of the subgroup
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
        const uint32_t o = __shfl_xor_sync(0xffffffffu, e, m);
        e = o > e ? o : e;
    }
    // x' = x * 2^(254 - bits*k - E) (k: position in the 16-bit half) or
    // x'' = x * 2^(238 - bits*j - E) (j: position in the byte); elements more
    // than 231 binades below E become a zero of their sign. For a normal x
    // within those 231 binades the scaled exponent field stays in [1, 254]
    // (at the extreme, 238 - 6 - 231 = 1), so the product is an integer add
    // to the exponent field; otherwise (zeros, subnormals, dropped elements)
    // it is formed with two exact power-of-two multiplies.
    uint32_t xr[8];
    if (emin >= 1 && int(e) - int(emin) <= 231) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = BF16_FIELDS ? (BITS == 4 ? (i & 1) : (i & 3)) : (BITS == 4 ? (i & 3) : i);
            const int pw = (BF16_FIELDS ? 238 : 254) - BITS * k - int(e);
            xr[i] = bits[i] + (uint32_t(pw) << 7);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = BF16_FIELDS ? (BITS == 4 ? (i & 1) : (i & 3)) : (BITS == 4 ? (i & 3) : i);
            const int pw = (BF16_FIELDS ? 238 : 254) - BITS * k - int(e);
            const int p1 = pw < 127 ? pw : 127;
            const float m1 = __uint_as_float(uint32_t(p1 + 127) << 23);
            const float m2 = __uint_as_float(uint32_t(pw - p1 + 127) << 23);
            const float r = int(e) - int((bits[i] >> 7) & 0xFFu) > 231 ? __uint_as_float((bits[i] & 0x8000u) << 16)
                                                                        : bf16_round(__fmul_rn(__fmul_rn(xv[i], m1), m2));
            xr[i] = __float_as_uint(r) >> 16;
        }
    }
    packed = make_uint4((xr[0] & 0xFFFFu) | (xr[1] << 16), (xr[2] & 0xFFFFu) | (xr[3] << 16),
                        (xr[4] & 0xFFFFu) | (xr[5] << 16), (xr[6] & 0xFFFFu) | (xr[7] << 16));
    // eight-element sum, left to right; the subgroup's sum gathers the eight in order
    float s8 = xv[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) s8 = __fadd_rn(s8, xv[i]);
    float sx = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float o = __shfl_sync(0xffffffffu, s8, i, 8);
        sx = i == 0 ? o : __fadd_rn(sx, o);
    }
    const int c = int(e) - 105;  // f1 * f2 = 2^c
    const int c1 = c < 127 ? c : 127;
    meta = make_float4(sx, __uint_as_float(uint32_t(c1 + 127) << 23), __uint_as_float(uint32_t(c - c1 + 127) << 23),
                       0.0f);
}

// Octet position of eighth e8 of subgroup t in processing order.
template <int BITS>
__device__ __forceinline__ int octet_position(int t, int e8)
{
    return BITS == 4 ? (e8 ^ (((t >> 2) & 1) * 4)) : e8;
}

// Writes eighth e8 of subgroup t (its staged x' and, from e8 = 0, the
// subgroup's (sx, f1, f2, 0)) into the streamed kernel's kXsF32-byte cell:
// its 64 x' (octets in processing order) as fp32 -- exactly the bf16 values,
// so the datapath unpacks nothing -- then the meta.
template <int BITS>
__device__ __forceinline__ void write_cell(uint8_t *cell, int t, int e8, const uint4 &packed, const float4 &meta)
{
    uint4 *dst = reinterpret_cast<uint4 *>(cell + octet_position<BITS>(t, e8) * 32);
    dst[0] = make_uint4(packed.x << 16, packed.x & 0xFFFF0000u, packed.y << 16, packed.y & 0xFFFF0000u);
    dst[1] = make_uint4(packed.z << 16, packed.z & 0xFFFF0000u, packed.w << 16, packed.w & 0xFFFF0000u);
    if (e8 == 0) *reinterpret_cast<float4 *>(cell + 256) = meta;
}

// Steps 1 and 2 for every vector, once per call, for the streamed kernel:
// cell (v, t) of vector v and subgroup t at out + (v * S_row + t) * cell
// bytes. Eight threads per subgroup (the grid is a whole number of warps;
// threads past the end only take part in the shuffles).
template <int BITS>
__device__ __forceinline__ void stage_all_body(const uint16_t *x, int K, int S_row, int V, uint8_t *out,
                                               unsigned *counters, int ncounters)
{
    grid_launch_dependents();  // the streamed kernel may start loading weights
    grid_dependency_wait();    // x may be written by the preceding grid
    // the K-split tickets of the streamed kernel start at zero
    for (int i = int(blockIdx.x) * int(blockDim.x) + int(threadIdx.x); i < ncounters; i += int(gridDim.x * blockDim.x))
        counters[i] = 0u;
    const int per_vec = S_row * 8, all = V * per_vec;
    const int u = int(blockIdx.x) * int(blockDim.x) + int(threadIdx.x);
    const bool live = u < all;  // uniform over each eight-lane group
    const int v = live ? u / per_vec : 0;
    const int rem = live ? u - v * per_vec : 0;
    const int t = rem >> 3, e8 = rem & 7;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (live) raw = __ldg(reinterpret_cast<const uint4 *>(x + size_t(v) * K + size_t(t) * kSub) + e8);
    uint4 packed;
    float4 meta;
    stage_eight<BITS, false>(raw, packed, meta);
    if (live) write_cell<BITS>(out + (size_t(v) * S_row + t) * kXsF32, t, e8, packed, meta);
}

// Stages x (one vector) for the ring kernel: the raw bf16 x of subgroups
// [sub_lo, sub_lo + nsub) lies densely at xr (128 bytes a subgroup, landed by
// one bulk copy); subgroup sl gets a kXsB16-byte cell at xc + kXsB16 * sl, its
// x'' with octet o (processing order) at 16 * o, then its (sx, f1, f2, 0).
// The 16 bytes past each 128 put the same octet of 32 consecutive cells on
// different banks.
template <int BITS>
__device__ __forceinline__ void stage_x_cells(uint32_t xr, uint32_t xc, int sub_lo, int nsub, int tid, int nthreads)
{
    const int all = nsub * 8;
    const int all_pad = (all + nthreads - 1) / nthreads * nthreads;
    for (int u = tid; u < all_pad; u += nthreads) {
        const bool live = u < all;  // uniform over each eight-lane group
        const int sl = live ? u >> 3 : 0, e8 = u & 7;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (live) raw = lds_v4_u32(xr + uint32_t(sl) * 128u + uint32_t(e8) * 16u);
        uint4 packed;
        float4 meta;
        stage_eight<BITS, true>(raw, packed, meta);
        if (live) {
            const uint32_t cell = xc + uint32_t(sl) * uint32_t(kXsB16);
            sts_v4_u32(cell + uint32_t(octet_position<BITS>(sub_lo + sl, e8)) * 16u, packed);
            if (e8 == 0) sts_v4_u32(cell + 128u, make_uint4(__float_as_uint(meta.x), __float_as_uint(meta.y),
                                                            __float_as_uint(meta.z), 0u));
        }
    }
}

// One chunk of one vector for 4 rows (steps 1 to 3): the lane's subgroup
// from `quads`, its x'' at xsub (swizzle sw) and (sx, f1, f2) at xmeta;
// returns the chunk value of row
// lane >> 3 (all lanes of that row's eight-lane group hold it).
template <int BITS, bool SWZ = true>
__device__ __forceinline__ float chunk_v1(const uint4 (&quads)[kRows][BITS == 4 ? 2 : 1], uint32_t xsub, uint32_t sw,
                                          uint32_t xmeta, const float (&fs)[kRows], const float (&fb)[kRows], bool active,
                                          int lane)
{
    float ae[kRows], ao[kRows];
    subgroup_dot_v1<BITS, SWZ>(quads, xsub, sw, ae, ao);
    const float4 meta = lds_f4(xmeta);
    float val[4];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        const float term = subgroup_term<false>(ae[r], ao[r], fs[r], fb[r], meta.x, meta.y, meta.z);
        val[r] = active ? term : 0.0f;
    }
    return tree_reduce_scatter<4>(val, lane);
}

// Step 4 and the output: fold the chunk values of the CTA's rows (cvs, laid
// out [row][chunk][vector]) left to right into y -- directly when the CTA
// covers all chunks, else through the workspace, the CTA that completes a row
// range last folding all chunks. Every partial it reads was written by this
// call; the range's ticket counter starts at zero (the launch clears it) and
// returns to zero.
template <int V>
__device__ __forceinline__ void fold_chunks(const float *cvs, int nrows, int row_t0, int c_lo, int cpc_here, int rb_lo,
                                            int tid, int nthreads, int N, int ks, int cpc, float *partials,
                                            unsigned *counters, void *y, int f32_out)
{
    __shared__ unsigned s_ticket;
    auto store_y = [&](int v, int n, float val) {
        if (f32_out)
            static_cast<float *>(y)[size_t(v) * N + n] = val;
        else
            static_cast<__nv_bfloat16 *>(y)[size_t(v) * N + n] = __float2bfloat16_rn(val);
    };
    if (cpc >= ks) {
        for (int idx = tid; idx < nrows * V; idx += nthreads) {
            const int v = idx / nrows, r = idx - v * nrows;
            const int n = row_t0 + r;
            if (n >= N) continue;
            float acc = cvs[(r * cpc_here) * V + v];
            for (int c = 1; c < ks; ++c) acc = __fadd_rn(acc, cvs[(r * cpc_here + c) * V + v]);
            store_y(v, n, acc);
        }
        return;
    }
    for (int idx = tid; idx < nrows * V * cpc_here; idx += nthreads) {
        const int cl = idx / (nrows * V), rem = idx - cl * nrows * V;
        const int v = rem / nrows, r = rem - v * nrows;
        const int n = row_t0 + r;
        if (n < N) __stcg(partials + (size_t(c_lo + cl) * V + v) * N + n, cvs[(r * cpc_here + cl) * V + v]);
    }
    __threadfence();
    __syncthreads();
    const unsigned nranges = unsigned(gridDim.y);
    if (tid == 0) s_ticket = atomicInc(counters + rb_lo, nranges - 1);
    __syncthreads();
    if (s_ticket != nranges - 1) return;
    __threadfence();
    // The fold of every (vector, row) of the range, left to right over the
    // ks chunk values: kU items per thread and up to kC chunks of each are
    // loaded before they are added, so the round trips overlap.
    constexpr int kU = 8, kC = 4;
    const size_t plane = size_t(V) * N;
    for (int base = tid; base < nrows * V; base += nthreads * kU) {
        size_t off[kU];
        bool ok[kU];
        float acc[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int idx = base + u * nthreads;
            const int v = idx / nrows, r = idx - v * nrows;
            ok[u] = idx < nrows * V && row_t0 + r < N;
            off[u] = ok[u] ? size_t(v) * N + size_t(row_t0 + r) : 0;
            acc[u] = 0.0f;
        }
        for (int c0 = 0; c0 < ks; c0 += kC) {
            float t[kC][kU];
#pragma unroll
            for (int c = 0; c < kC; ++c)
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    t[c][u] = ok[u] && c0 + c < ks ? __ldcg(partials + size_t(c0 + c) * plane + off[u]) : 0.0f;
#pragma unroll
            for (int c = 0; c < kC; ++c)
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    if (c0 + c < ks) acc[u] = c0 + c == 0 ? t[c][u] : __fadd_rn(acc[u], t[c][u]);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (!ok[u]) continue;
            const int idx = base + u * nthreads;
            const int v = idx / nrows;
            store_y(v, int(off[u] - size_t(v) * N), acc[u]);
        }
    }
}

// ------------------------------------------------------- one vector: ring --

template <int BITS, int GS, bool SBP, int V = 1>
__device__ __forceinline__ void qmv_ring_body(const CUtensorMap *map_w, const CUtensorMap *map_s, const CUtensorMap *map_b,
                                              const RingParams &p)
{
    constexpr int kSubB = sub_bytes(BITS);
    constexpr int kChunkB = chunk_bytes(BITS);
    constexpr int NP = BITS == 4 ? 2 : 1;

    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;
    const int C = p.consumers;
    const int P = nwarps - C;

    const int c_lo = blockIdx.y * p.cpc;
    const int c_hi = c_lo + p.cpc < p.ks ? c_lo + p.cpc : p.ks;
    const int sub_lo = c_lo * kChunkSubs;
    const int sub_hi = c_hi * kChunkSubs < p.S_row ? c_hi * kChunkSubs : p.S_row;
    const int nsub = sub_hi - sub_lo;
    const int rb_lo = int((long long)blockIdx.x * p.NB / p.grid_rows);
    const int rb_hi = int((long long)(blockIdx.x + 1) * p.NB / p.grid_rows);
    const int row_t0 = rb_lo * kRows;
    const int cpc_here = c_hi - c_lo;
    const int upr = (cpc_here + p.uc - 1) / p.uc;  // units per row block
    const int nunits = (rb_hi - rb_lo) * upr;

    const int nsub_max = p.cpc * kChunkSubs < p.S_row ? p.cpc * kChunkSubs : p.S_row;
    const RingLayout L = ring_layout(p.pitch, p.sb_mode_unit, p.sbox, SBP, p.slots, nsub_max, p.max_rb, p.cpc, V);
    // metadata: bytes per element (a bf16, or an interleaved scale|bias pair)
    // and the box start alignment in elements (16 bytes)
    constexpr int sbE = sb_elem_bytes(SBP), sbA = 16 / sbE;
    const uint32_t ring = smem_u32(smem + L.ring);
    const uint32_t xr = smem_u32(smem + L.xr), xc = smem_u32(smem + L.xc);
    float *cvs = reinterpret_cast<float *>(smem + L.cv);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar);  // full[slots], empty[slots], x
    unsigned *s_next = reinterpret_cast<unsigned *>(smem + L.misc);
    volatile unsigned *s_abort = s_next + 1;
    // s_issued[k]: units issued by producer k (it issues k, k + P, ...).
    volatile int *s_issued = reinterpret_cast<volatile int *>(s_next + 2);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + p.slots), xbar = smem_u32(bars + 2 * p.slots);

    // Geometry of unit u: rows [r0, r0 + nr), chunks [c0, c1).
    struct Unit {
        int r0, nr, c0, c1;
    };
    auto unit_geo = [&](int u) {
        Unit g;
        const int rbl = u / upr, pc = u - rbl * upr;
        g.r0 = (rb_lo + rbl) * kRows;
        g.nr = p.N - g.r0 < kRows ? p.N - g.r0 : kRows;
        g.c0 = c_lo + pc * p.uc;
        g.c1 = g.c0 + p.uc < c_hi ? g.c0 + p.uc : c_hi;
        return g;
    };
    // Element coordinate of metadata box `bx` of a unit (rows r0.., groups from chunk c0).
    auto sb_coord = [&](const Unit &g, int bx) {
        const long long g0 = (long long)g.c0 * kChunkElems / GS;
        return int(((long long)(g.r0 + bx) * p.G + g0) & ~(long long)(sbA - 1));
    };

    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](const Unit &g, int slot) {
        const uint32_t base = ring + slot * L.slot_bytes;
        const uint32_t full = full0 + 8 * slot;
        const int e0 = g.c0 * kChunkElems;
        const int e1 = g.c1 * kChunkElems < p.K ? g.c1 * kChunkElems : p.K;
        const uint32_t seg = uint32_t(e1 - e0) * BITS / 8;
        if (p.unit_mode == kUnitTiles) {
            // boxes of 4 rows: rows past N and bytes past the row's end arrive as zeros
            mbar_arrive_expect_tx(full, uint32_t(kRows * p.pitch + (SBP ? 1 : 2) * p.sbox * sbE));
            tma_load_2d_hint(base, map_w, g.c0 * (kChunkB / 8), g.r0, full, pol);
            tma_load_2d(base + L.sb_off, map_s, g.c0 * (kChunkElems / GS), g.r0, full);
            if constexpr (!SBP) tma_load_2d(base + L.sb_off + L.sbs, map_b, g.c0 * (kChunkElems / GS), g.r0, full);
            return;
        }
        const int nbox = p.sb_mode_unit ? 1 : g.nr;
        const uint32_t wbytes = p.unit_mode == kUnitRows ? uint32_t(g.nr) * uint32_t(p.row_bytes) : uint32_t(g.nr) * seg;
        mbar_arrive_expect_tx(full, wbytes + uint32_t((SBP ? 1 : 2) * nbox * p.sbox * sbE));
        if (p.unit_mode == kUnitRows) {
            bulk_load(base, p.w + size_t(g.r0) * p.row_bytes, wbytes, full, pol);
        } else {
            for (int r = 0; r < g.nr; ++r)
                bulk_load(base + r * p.pitch, p.w + size_t(g.r0 + r) * p.row_bytes + size_t(e0) * BITS / 8, seg, full,
                          pol);
        }
        for (int bx = 0; bx < nbox; ++bx) {
            const int xc = sb_coord(g, bx);
            tma_load_1d(base + L.sb_off + bx * L.sbs, map_s, xc, full);
            if constexpr (!SBP) tma_load_1d(base + L.sb_off + (nbox + bx) * L.sbs, map_b, xc, full);
        }
    };

    // The ring protocol needs every slot served by one producer and consumed
    // by one consumer warp: slots a multiple of both counts.
    if (C > p.slots || C < 1 || P < 1 || p.slots % P != 0 || p.slots % C != 0) {
        if (tid == 0) atomicOr(p.err, 2u);
        return;
    }
    if (tid < 2 * p.slots + 1) {  // full[], empty[] and the x barrier are contiguous
        mbar_init(full0 + 8 * tid, 1);
        fence_mbar_init();
    }
    if (tid == 0) {
        *s_next = 0;
        *s_abort = 0;
    }
    if (tid < P) s_issued[tid] = 0;
    __syncthreads();
    grid_launch_dependents();

    if (warp >= C) {
        // --------------------------------------------------------- producers
        // Producer k issues units k, k + P, ... (so it alone serves the slots
        // congruent to k modulo P), each after the slot's previous unit was
        // consumed. The launch may overlap the preceding grid: unless the
        // caller allowed weights to be read under it, the producers wait for it
        // before their first copy.
        if (!p.early_weights) grid_dependency_wait();
        const int kp = warp - C;
        bool ok = true;
        int slot = kp, lap = 0, rbl = 0, pc = kp;
        while (pc >= upr) {
            pc -= upr;
            ++rbl;
        }
        for (int u = kp; u < nunits; u += P) {
            if (lane == 0) {
                if (lap > 0) ok = !*s_abort && mbar_wait_bounded(empty0 + 8 * slot, (lap - 1) & 1);
                if (ok) {
                    Unit g;
                    g.r0 = (rb_lo + rbl) * kRows;
                    g.nr = p.N - g.r0 < kRows ? p.N - g.r0 : kRows;
                    g.c0 = c_lo + pc * p.uc;
                    g.c1 = g.c0 + p.uc < c_hi ? g.c0 + p.uc : c_hi;
                    issue(g, slot);
                    __threadfence_block();
                    s_issued[kp] = u + 1;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            slot += P;
            if (slot >= p.slots) {
                slot -= p.slots;
                ++lap;
            }
            pc += P;
            while (pc >= upr) {
                pc -= upr;
                ++rbl;
            }
        }
        if (!ok && lane == 0) {
            atomicOr(p.err, 1u);
            *s_abort = 1;
        }
    } else {
        // --------------------------------------------------------- consumers
        // Consumer warp c takes units c, c + C, ...; with the slot count a
        // multiple of C, slot s is only ever consumed by warp s % C, in unit
        // order, so a unit's data is announced by its slot's phase parity
        // alone: the producer refills a slot only after its one consumer has
        // released the unit before.
        grid_dependency_wait();  // x may be written by the preceding grid
        if constexpr (V == 1) {
            if (tid == 0) {
                // the CTA's x range in one copy, landing where it is staged from
                mbar_arrive_expect_tx(xbar, uint32_t(nsub) * 128u);
                bulk_load_plain(xr, p.x + size_t(sub_lo) * kSub, uint32_t(nsub) * 128u, xbar);
            }
        } else {
            if (tid == 0) {
                // the call's staged cells of this CTA's range, one copy per vector
                mbar_arrive_expect_tx(xbar, uint32_t(V * nsub) * kXsF32);
                for (int v = 0; v < V; ++v)
                    bulk_load_plain(xc + uint32_t(v * nsub) * kXsF32, p.xs_staged + (size_t(v) * p.S_row + sub_lo) * kXsF32,
                                    uint32_t(nsub) * kXsF32, xbar);
            }
        }
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(xbar, 0)) && lane == 0) {
            atomicOr(p.err, 1u);
            *s_abort = 1;
        }
        if constexpr (V == 1) stage_x_cells<BITS>(xr, xc, sub_lo, nsub, tid, C * 32);
        asm volatile("bar.sync 1, %0;" ::"r"(C * 32) : "memory");  // consumer warps only

        uint32_t poff[NP];
        piece_offsets<BITS>(lane, poff);
        int slot = warp, lap = 0;
        for (int u = warp; u < nunits; u += C) {
            bool ok = !*s_abort;
            if (ok) ok = mbar_wait_bounded(full0 + 8 * slot, lap & 1);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) {
                    atomicOr(p.err, 1u);
                    *s_abort = 1;
                }
                break;
            }
            const Unit g = unit_geo(u);
            const uint32_t base = ring + slot * L.slot_bytes;
            const int nbox = p.sb_mode_unit ? 1 : g.nr;
            // Per-unit shared addresses of row r's scale / bias (or pair) of
            // group 0 of the row (rows past N alias row 0).
            uint32_t sa[kRows], ba[kRows];
            if (p.unit_mode == kUnitTiles) {
                // box rows of sbox / 4 groups starting at the unit's first group
                const int gb = p.sbox / kRows, g0 = g.c0 * (kChunkElems / GS);
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    sa[r] = base + L.sb_off + uint32_t(sbE * (r * gb - g0));
                    ba[r] = sa[r] + L.sbs;
                }
            } else {
                const int g0 = g.c0 * (kChunkElems / GS);
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    const int rr = r < g.nr ? r : 0;
                    const int bx = p.sb_mode_unit ? 0 : rr;
                    // N * G < 2^31: element indices fit 32 bits
                    const int xst = ((g.r0 + bx) * p.G + g0) & ~(sbA - 1);
                    sa[r] = base + L.sb_off + bx * L.sbs + sbE * ((g.r0 + rr) * p.G - xst);
                    ba[r] = sa[r] + nbox * L.sbs;
                }
            }
            for (int cc = g.c0; cc < g.c1; ++cc) {
                const int t = cc * kChunkSubs + lane;        // subgroup index in the row
                const bool active = t < p.S_row;
                const int tl = active ? t : cc * kChunkSubs;  // a staged subgroup for idle lanes
                // lanes past the row's end read subgroup 0 of the chunk (discarded)
                const uint32_t coff = uint32_t((cc - g.c0) * kChunkB) - (active ? 0u : uint32_t(lane) * kSubB);
                uint4 quads[kRows][NP];
#pragma unroll
                for (int r = 0; r < kRows; ++r)
#pragma unroll
                    for (int pc = 0; pc < NP; ++pc)
                        quads[r][pc] = lds_v4_u32(base + uint32_t(r * p.pitch) + coff + poff[pc]);
                // byte offset of the lane's group in a row's metadata
                const uint32_t go = uint32_t(tl * (kSub / 32) / (GS / 32)) * uint32_t(sbE);
                float fs[kRows], fb[kRows];
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    if constexpr (SBP) {  // one pair: scale in the low half, bias in the high half
                        const uint32_t v = lds_u32(sa[r] + go);
                        fs[r] = __uint_as_float(v << 16);
                        fb[r] = __uint_as_float(v & 0xFFFF0000u);
                    } else {
                        fs[r] = bf16_bits_to_f32(lds_u16(sa[r] + go));
                        fb[r] = bf16_bits_to_f32(lds_u16(ba[r] + go));
                    }
                }
                if constexpr (V == 1) {
                    const uint32_t cell = xc + uint32_t(tl - sub_lo) * uint32_t(kXsB16);
                    const float tot = chunk_v1<BITS, false>(quads, cell, 0u, cell + 128u, fs, fb, active, lane);
                    const int r = lane >> 3;
                    if ((lane & 7) == 0 && r < g.nr) cvs[(g.r0 - row_t0 + r) * cpc_here + (cc - c_lo)] = tot;
                } else {
                    // V vectors: fp32 cells, packed fmas (the streamed kernel's datapath)
                    constexpr int NVAL = kRows * V;
                    constexpr int NRED = NVAL <= 4 ? 4 : NVAL <= 8 ? 8 : NVAL <= 16 ? 16 : 32;
                    const uint32_t xv_bytes = uint32_t(nsub) * kXsF32;
                    const uint32_t xsub = xc + uint32_t(tl - sub_lo) * kXsF32;
                    uint64_t acc[kRows][V];
                    subgroup_dot_vp<BITS, V>(quads, xsub, xv_bytes, acc);
                    float val[NRED];
#pragma unroll
                    for (int i = 0; i < NRED; ++i) val[i] = 0.0f;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const float4 meta = lds_f4(xsub + v * xv_bytes + 256);
#pragma unroll
                        for (int r = 0; r < kRows; ++r) {
                            const float term = subgroup_term<true>(pair_lo(acc[r][v]), pair_hi(acc[r][v]), fs[r], fb[r], meta.x, meta.y, meta.z);
                            val[r * V + v] = active ? term : 0.0f;
                        }
                    }
                    const float tot = tree_reduce_scatter<NRED>(val, lane);
                    constexpr int SH = NRED == 4 ? 3 : NRED == 8 ? 2 : NRED == 16 ? 1 : 0;
                    const int idx = lane >> SH;
                    const int r = idx / V, v = idx - r * V;
                    if ((lane & ((1 << SH) - 1)) == 0 && idx < NVAL && r < g.nr)
                        cvs[((g.r0 - row_t0 + r) * cpc_here + (cc - c_lo)) * V + v] = tot;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);
            slot += C;
            if (slot >= p.slots) {
                slot -= p.slots;
                ++lap;
            }
        }
    }
    __syncthreads();
    if (*s_abort) {
        // Wait (bounded) for every copy this CTA may still have in flight.
        if (warp >= C && lane == 0) {
            const int kp = warp - C;
            const int hi = s_issued[kp];
            for (int u = hi - p.slots > kp ? hi - p.slots : kp; u < hi; u += P)
                (void)mbar_wait_bounded(full0 + 8 * (u % p.slots), (u / p.slots) & 1);
        }
        if (tid == 0) (void)mbar_wait_bounded(xbar, 0);  // the x copy
        __syncthreads();
        return;
    }
    fold_chunks<V>(cvs, (rb_hi - rb_lo) * kRows, row_t0, c_lo, cpc_here, rb_lo, tid, nthreads, p.N, p.ks, p.cpc,
                   p.partials, p.counters, p.y, p.f32_out);
}

// ------------------------------------------------ one vector: direct loads --

// Stages x (one vector) for qmv_one from global memory: subgroup sl of the
// CTA's range [sub_lo, sub_lo + nsub) gets a kXsB16-byte cell at
// xs + kXsB16 * sl: its x'' with octet o (processing order) at 16 * o, then
// its (sx, f1, f2, 0). The 16 bytes past each 128 put the same octet of 32
// consecutive cells on different banks.
template <int BITS>
__device__ __forceinline__ void stage_x_one(const uint16_t *x, uint32_t xs, int sub_lo, int nsub, int tid, int nthreads)
{
    const int all = nsub * 8;
    const int all_pad = (all + nthreads - 1) / nthreads * nthreads;
    for (int u = tid; u < all_pad; u += nthreads) {
        const bool live = u < all;  // uniform over each eight-lane group
        const int sl = live ? u >> 3 : 0, e8 = u & 7;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (live) raw = __ldg(reinterpret_cast<const uint4 *>(x + size_t(sub_lo + sl) * kSub) + e8);
        uint4 packed;
        float4 meta;
        stage_eight<BITS, true>(raw, packed, meta);
        if (live) {
            const uint32_t cell = xs + uint32_t(sl) * uint32_t(kXsB16);
            sts_v4_u32(cell + uint32_t(octet_position<BITS>(sub_lo + sl, e8)) * 16u, packed);
            if (e8 == 0) sts_v4_u32(cell + 128u, make_uint4(__float_as_uint(meta.x), __float_as_uint(meta.y),
                                                            __float_as_uint(meta.z), 0u));
        }
    }
}

// The one-vector kernel. CTA (i, j) owns row blocks [rb_lo, rb_hi) and chunks
// [c_lo, c_hi); its units are the (row block, chunk) pairs in row-block-major
// order. Warp w computes units w, w + W, ... (W warps): it loads a unit's
// weights (the lane's subgroup of 4 rows, two or one 16-byte loads per row),
// scales and biases straight into registers, and issues the next unit's loads
// before computing the current one. The first unit's loads go out before the
// wait for the preceding grid: weights, scales and biases never depend on it.
// Unit bookkeeping is incremental (no division per unit): the kernel issues
// about 1.7 instructions per weight in its datapath, which is what bounds it.
template <int BITS, int GS, bool SBP>
__device__ __forceinline__ void qmv_one_body(const Params &p)
{
    constexpr int kSubB = sub_bytes(BITS);
    constexpr int NP = BITS == 4 ? 2 : 1;

    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;

    const int c_lo = blockIdx.y * p.cpc;
    const int c_hi = c_lo + p.cpc < p.ks ? c_lo + p.cpc : p.ks;
    const int sub_lo = c_lo * kChunkSubs;
    const int sub_hi = c_hi * kChunkSubs < p.S_row ? c_hi * kChunkSubs : p.S_row;
    const int nsub = sub_hi - sub_lo;
    const int rb_lo = int((long long)blockIdx.x * p.NB / p.grid_rows);
    const int rb_hi = int((long long)(blockIdx.x + 1) * p.NB / p.grid_rows);
    const int nrb = rb_hi - rb_lo;
    const int row_t0 = rb_lo * kRows;
    const int cpc_here = c_hi - c_lo;

    const int nsub_max = p.cpc * kChunkSubs < p.S_row ? p.cpc * kChunkSubs : p.S_row;
    const OneLayout L = one_layout(nsub_max, p.max_rb, p.cpc);
    const uint32_t xs = smem_u32(smem + L.xs);
    float *cvs = reinterpret_cast<float *>(smem + L.cv);

    // Unit stepping: (rbl, ccl) = unit u of the CTA, advanced by W units at a
    // time (dr row blocks and dc chunks, one more row block on a carry). The
    // lane's byte offset of a unit's row 0 piece and the element index of its
    // row 0 metadata advance by fixed deltas, so no unit needs a multiply.
    const int dr = nwarps / cpc_here, dc = nwarps - dr * cpc_here;
    const long long rbB = (long long)kRows * p.row_bytes;  // bytes of one row block
    const long long wstep0 = dr * rbB + (long long)dc * chunk_bytes(BITS);
    const long long wstep1 = wstep0 + rbB - (long long)cpc_here * chunk_bytes(BITS);
    const int rbG = kRows * p.G;  // metadata elements of one row block (N * G < 2^31)
    constexpr int kGpc = kChunkElems / GS;  // groups per chunk
    const int estep0 = dr * rbG + dc * kGpc, estep1 = estep0 + rbG - cpc_here * kGpc;
    // Per lane: the offset of its first piece inside a subgroup row (4-bit:
    // the half selected by bit 2 of the lane, i.e. of the subgroup index,
    // first) and of the second; the last subgroup of a row for clamping.
    const int first = BITS == 4 ? ((lane >> 2) & 1) * 16 : 0;
    const int second = 16 - first;
    const int t_last = p.S_row - 1;
    const int sub_off = lane * kSubB;  // the lane's subgroup inside a chunk row

    int rbl = warp / cpc_here, ccl = warp - (warp / cpc_here) * cpc_here;
    // byte offset of the unit's chunk row 0 and element index of its row 0
    // metadata, without the lane's subgroup
    long long wo = (long long)(rb_lo + rbl) * rbB + (long long)(c_lo + ccl) * chunk_bytes(BITS);
    int eo = (rb_lo + rbl) * rbG + (c_lo + ccl) * kGpc;

    // Loads of the unit at (wo, eo), chunk ccl, row block rbl. Rows past N
    // re-read row 0 of the block and subgroups past the row's end re-read the
    // row's last subgroup (their results are discarded).
    auto load_unit = [&](long long wo_u, int eo_u, int rbl_u, int ccl_u, uint4 (&wq)[kRows][NP], uint32_t (&sv)[kRows],
                         uint32_t (&bv)[kRows]) {
        const int t = (c_lo + ccl_u) * kChunkSubs + lane;
        const int clamp = t > t_last ? t - t_last : 0;  // subgroups to step back
        const int nr = p.N - (rb_lo + rbl_u) * kRows;
        const uint8_t *w0 = p.w + wo_u + (sub_off - clamp * kSubB);
        const int e0 = eo_u + ((lane - clamp) * (kSub / 32)) / (GS / 32);
        if (nr >= kRows) {
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const uint8_t *wr = w0 + r * (long long)p.row_bytes;
                wq[r][0] = __ldcs(reinterpret_cast<const uint4 *>(wr + first));
                if constexpr (NP == 2) wq[r][1] = __ldcs(reinterpret_cast<const uint4 *>(wr + second));
                const int e = e0 + r * p.G;
                if constexpr (SBP) {  // one pair: scale in the low half, bias in the high half
                    const uint32_t v = __ldcs(reinterpret_cast<const unsigned int *>(p.scales) + e);
                    sv[r] = v & 0xFFFFu;
                    bv[r] = v >> 16;
                } else {
                    sv[r] = __ldcs(reinterpret_cast<const unsigned short *>(p.scales) + e);
                    bv[r] = __ldcs(reinterpret_cast<const unsigned short *>(p.biases) + e);
                }
            }
        } else {
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const int ro = r < nr ? r : 0;
                const uint8_t *wr = w0 + ro * (long long)p.row_bytes;
                wq[r][0] = __ldcs(reinterpret_cast<const uint4 *>(wr + first));
                if constexpr (NP == 2) wq[r][1] = __ldcs(reinterpret_cast<const uint4 *>(wr + second));
                const int e = e0 + ro * p.G;
                if constexpr (SBP) {
                    const uint32_t v = __ldcs(reinterpret_cast<const unsigned int *>(p.scales) + e);
                    sv[r] = v & 0xFFFFu;
                    bv[r] = v >> 16;
                } else {
                    sv[r] = __ldcs(reinterpret_cast<const unsigned short *>(p.scales) + e);
                    bv[r] = __ldcs(reinterpret_cast<const unsigned short *>(p.biases) + e);
                }
            }
        }
    };
    // Steps 1-3 of unit (rbl_u, ccl_u) from its registers; its chunk value of
    // row lane >> 3 goes to shared memory.
    auto compute_unit = [&](int rbl_u, int ccl_u, const uint4 (&wq)[kRows][NP], const uint32_t (&sv)[kRows],
                            const uint32_t (&bv)[kRows]) {
        const int t = (c_lo + ccl_u) * kChunkSubs + lane;
        const bool active = t <= t_last;
        const uint32_t sl = uint32_t((active ? t : t_last) - sub_lo);
        float fs[kRows], fb[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            fs[r] = bf16_bits_to_f32(sv[r]);
            fb[r] = bf16_bits_to_f32(bv[r]);
        }
        const uint32_t cell = xs + sl * uint32_t(kXsB16);
        const float tot = chunk_v1<BITS, false>(wq, cell, 0u, cell + 128u, fs, fb, active, lane);
        const int r = lane >> 3;
        if ((lane & 7) == 0 && r < p.N - (rb_lo + rbl_u) * kRows) cvs[(rbl_u * kRows + r) * cpc_here + ccl_u] = tot;
    };
    auto advance = [&](int &rb_u, int &cc_u, long long &wo_u, int &eo_u) {
        cc_u += dc;
        rb_u += dr;
        const bool carry = cc_u >= cpc_here;
        if (carry) {
            cc_u -= cpc_here;
            ++rb_u;
        }
        wo_u += carry ? wstep1 : wstep0;
        eo_u += carry ? estep1 : estep0;
    };


    // Two register sets, A and B, alternate: while one unit is computed the
    // next one's loads are in flight.
    uint4 wa[kRows][NP], wb[kRows][NP];
    uint32_t sa[kRows] = {0, 0, 0, 0}, ba[kRows] = {0, 0, 0, 0}, sb[kRows] = {0, 0, 0, 0}, bb[kRows] = {0, 0, 0, 0};
    if (!p.early_weights) grid_dependency_wait();  // the launch may overlap the preceding grid
    if (rbl < nrb) load_unit(wo, eo, rbl, ccl, wa, sa, ba);
    grid_launch_dependents();
    grid_dependency_wait();  // x may be written by the preceding grid
    stage_x_one<BITS>(p.x, xs, sub_lo, nsub, tid, nthreads);
    __syncthreads();

    while (rbl < nrb) {
        int rb1 = rbl, cc1 = ccl, eo1 = eo;
        long long wo1 = wo;
        advance(rb1, cc1, wo1, eo1);
        if (rb1 < nrb) load_unit(wo1, eo1, rb1, cc1, wb, sb, bb);
        compute_unit(rbl, ccl, wa, sa, ba);
        if (rb1 >= nrb) break;
        rbl = rb1;
        ccl = cc1;
        wo = wo1;
        eo = eo1;
        advance(rb1, cc1, wo1, eo1);
        if (rb1 < nrb) load_unit(wo1, eo1, rb1, cc1, wa, sa, ba);
        compute_unit(rbl, ccl, wb, sb, bb);
        rbl = rb1;
        ccl = cc1;
        wo = wo1;
        eo = eo1;
    }
    __syncthreads();
    fold_chunks<1>(cvs, nrb * kRows, row_t0, c_lo, cpc_here, rb_lo, tid, nthreads, p.N, p.ks, p.cpc, p.partials,
                   p.counters, p.y, p.f32_out);
}

// ------------------------------------------------ V vectors: direct loads --

template <int BITS, int GS, int V, bool SBP>
__device__ __forceinline__ void qmv_direct_body(const Params &p)
{
    using T = Traits<BITS, V>;
    constexpr int kSubB = sub_bytes(BITS);

    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nthreads = blockDim.x;

    const int c_lo = blockIdx.y * p.cpc;
    const int c_hi = c_lo + p.cpc < p.ks ? c_lo + p.cpc : p.ks;
    const int sub_lo = c_lo * kChunkSubs;
    const int sub_hi = c_hi * kChunkSubs < p.S_row ? c_hi * kChunkSubs : p.S_row;
    const int nsub = sub_hi - sub_lo;
    const int rb_lo = int((long long)blockIdx.x * p.NB / p.grid_rows);
    const int rb_hi = int((long long)(blockIdx.x + 1) * p.NB / p.grid_rows);
    const int row_t0 = rb_lo * kRows;
    const int cpc_here = c_hi - c_lo;
    const int nunits = (rb_hi - rb_lo) * cpc_here;  // (row block, chunk) pairs

    const int nsub_max = p.cpc * kChunkSubs < p.S_row ? p.cpc * kChunkSubs : p.S_row;
    const SmemLayout L = smem_layout(BITS, V, nthreads >> 5, nsub_max, p.max_rb, p.cpc);
    const uint32_t xs = smem_u32(smem + L.xs);
    float *cvs = reinterpret_cast<float *>(smem + L.cv);
    unsigned *s_next = reinterpret_cast<unsigned *>(smem + L.misc);
    const uint32_t xbar = smem_u32(smem + L.misc + 8);
    if (tid == 0) {
        *s_next = 0;
        mbar_init(xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    uint32_t poff[T::NP];
    piece_offsets<BITS>(lane, poff);
    // The next work item for this warp (items are taken in increasing order).
    auto grab = [&]() {
        int u = 0;
        if (lane == 0) u = int(atomicAdd(s_next, 1u));
        return __shfl_sync(0xffffffffu, u, 0);
    };
    struct Unit {
        int r0, nr, cc, t, tc;  // rows [r0, r0 + nr), chunk cc, the lane's subgroup (tc: clamped into the row)
    };
    auto unit_geo = [&](int u) {
        Unit g;
        const int rbl = u / cpc_here;
        g.r0 = (rb_lo + rbl) * kRows;
        g.nr = p.N - g.r0 < kRows ? p.N - g.r0 : kRows;
        g.cc = c_lo + (u - rbl * cpc_here);
        g.t = g.cc * kChunkSubs + lane;
        g.tc = g.t < p.S_row ? g.t : p.S_row - 1;
        return g;
    };
    // Unit u's weight bytes of this lane (4 rows x its subgroup, pieces in
    // processing order), and the scale and bias of its group in each row.
    // Rows past N and subgroups past the row's end re-read valid bytes
    // (their results are discarded).
    auto load_unit = [&](int u, uint4 (&wq)[kRows][T::NP], uint32_t (&sv)[kRows], uint32_t (&bv)[kRows]) {
        const Unit g = unit_geo(u);
        const int gi = g.tc * (kSub / 32) / (GS / 32);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int row = g.r0 + (r < g.nr ? r : 0);
            const uint8_t *src = p.w + size_t(row) * p.row_bytes + size_t(g.tc) * kSubB;
#pragma unroll
            for (int pc = 0; pc < T::NP; ++pc)
                wq[r][pc] = __ldg(reinterpret_cast<const uint4 *>(src + (BITS == 4 ? (poff[pc] & 31u) : 0u)));
            const size_t e = size_t(row) * p.G + gi;
            if constexpr (SBP) {  // one pair: scale in the low half, bias in the high half
                const uint32_t v = __ldg(reinterpret_cast<const uint32_t *>(p.scales) + e);
                sv[r] = v & 0xFFFFu;
                bv[r] = v >> 16;
            } else {
                sv[r] = __ldg(p.scales + e);
                bv[r] = __ldg(p.biases + e);
            }
        }
    };

    // The first item's loads first: they do not depend on the preceding grid
    // (the call's staging kernel), so their latency overlaps it. Item i is
    // unit i / IPU, passes from (i % IPU) * PPI on.
    const int nitems = nunits * T::IPU;
    int i0 = grab();
    uint4 w_cur[kRows][T::NP];
    uint32_t s_cur[kRows] = {0, 0, 0, 0}, b_cur[kRows] = {0, 0, 0, 0};
    if (i0 < nitems) load_unit(i0 / T::IPU, w_cur, s_cur, b_cur);
    grid_launch_dependents();
    grid_dependency_wait();  // the staged cells are written by the preceding grid
    constexpr uint32_t kCell = kXsF32;
    if (tid == 0) {
        // this CTA's subgroups of every vector: one bulk copy per vector
        mbar_arrive_expect_tx(xbar, uint32_t(V * nsub) * kCell);
        for (int v = 0; v < V; ++v)
            bulk_load_plain(xs + uint32_t(v * nsub_max) * kCell, p.xs_staged + (size_t(v) * p.S_row + sub_lo) * kCell,
                            uint32_t(nsub) * kCell, xbar);
    }
    if (__syncthreads_or(!mbar_wait_bounded(xbar, 0))) {
        if (tid == 0) {
            atomicOr(p.err, 1u);
            (void)mbar_wait_bounded(xbar, 0);  // the copies may still be landing
        }
        __syncthreads();
        return;
    }

    const uint32_t xv_bytes = uint32_t(nsub_max) * kXsF32;
    const uint32_t wcell = smem_u32(smem + L.wbuf) + uint32_t(warp) * kRows * T::NP * 512u + uint32_t(lane) * 16u;
    while (i0 < nitems) {
        const int u0 = i0 / T::IPU, ps0 = (i0 - u0 * T::IPU) * T::PPI;
        const Unit g = unit_geo(u0);
        const bool active = g.t < p.S_row;
        const int sl = (active ? g.t : g.cc * kChunkSubs) - sub_lo;  // a staged subgroup for idle lanes
        float fs[kRows], fb[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            fs[r] = bf16_bits_to_f32(s_cur[r]);
            fb[r] = bf16_bits_to_f32(b_cur[r]);
        }
        // two passes in this item: park the weight bytes in this lane's cells
        // of the warp's buffer (only this lane reads them back)
        if constexpr (T::PPI > 1) {
#pragma unroll
            for (int r = 0; r < kRows; ++r)
#pragma unroll
                for (int pc = 0; pc < T::NP; ++pc) sts_v4_u32(wcell + uint32_t(r * T::NP + pc) * 512u, w_cur[r][pc]);
        }
#pragma unroll
        for (int pp = 0; pp < T::PPI; ++pp) {
            const int v0 = (ps0 + pp) * T::VP;
            const uint32_t xsub = xs + (uint32_t(v0) * nsub_max + sl) * kXsF32;
            uint64_t acc[kRows][T::VP];
            if constexpr (T::PPI > 1)
                subgroup_dot_vp_smem<BITS, T::VP>(wcell, xsub, xv_bytes, acc);
            else
                subgroup_dot_vp<BITS, T::VP>(w_cur, xsub, xv_bytes, acc);
            float val[T::NRED];
#pragma unroll
            for (int i = 0; i < T::NRED; ++i) val[i] = 0.0f;
#pragma unroll
            for (int v = 0; v < T::VP; ++v) {
                if (v0 + v >= V) break;
                const float4 meta = lds_f4(xsub + v * xv_bytes + 256);
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    const float term = subgroup_term<true>(pair_lo(acc[r][v]), pair_hi(acc[r][v]), fs[r], fb[r], meta.x, meta.y, meta.z);
                    val[r * T::VP + v] = active ? term : 0.0f;
                }
            }
            const float tot = tree_reduce_scatter<T::NRED>(val, lane);
            // lane holds value index lane >> (5 - log2 NRED)
            constexpr int SH = T::NRED == 4 ? 3 : T::NRED == 8 ? 2 : T::NRED == 16 ? 1 : 0;
            const int idx = lane >> SH;
            const int r = idx / T::VP, v = idx - r * T::VP;
            if ((lane & ((1 << SH) - 1)) == 0 && idx < T::NVAL && v0 + v < V && r < g.nr)
                cvs[((g.r0 - row_t0 + r) * cpc_here + (g.cc - c_lo)) * V + v0 + v] = tot;
        }
        // the next item: its loads are issued only now (the other warps'
        // arithmetic covers their latency)
        i0 = grab();
        if (i0 < nitems) load_unit(i0 / T::IPU, w_cur, s_cur, b_cur);
    }
    __syncthreads();
    fold_chunks<V>(cvs, (rb_hi - rb_lo) * kRows, row_t0, c_lo, cpc_here, rb_lo, tid, nthreads, p.N, p.ks, p.cpc,
                   p.partials, p.counters, p.y, p.f32_out);
}

// Launch bounds: the one-vector kernel runs at most 16 consumer warps and 4
// producer warps; the streamed kernel at most 12 warps (its registers go to
// the V-vector accumulators; at two or three vectors the plan may launch
// 8-warp CTAs, two per SM).
constexpr int kConsumersV1 = 16;
constexpr int kProducersV1 = 4;
constexpr int kThreadsV1 = (kConsumersV1 + kProducersV1) * 32;
constexpr int kThreadsVN = 12 * 32;

// SBP: scales and biases arrive interleaved (one 32-bit pair per group).
template <int BITS, int GS, bool SBP>
__global__ void __launch_bounds__(kThreadsV1, 1)
    qmv_m1(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_s,
           const __grid_constant__ CUtensorMap map_b, const RingParams p)
{
    qmv_ring_body<BITS, GS, SBP>(&map_w, &map_s, &map_b, p);
}

// The ring for 2..4 vectors (staged cells from the workspace): at most 12
// consumer warps and 4 producers, 128 registers.
constexpr int kThreadsRingV = 16 * 32;
template <int BITS, int GS, bool SBP, int V>
__global__ void __launch_bounds__(kThreadsRingV, 1)
    qmv_ringv(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_s,
              const __grid_constant__ CUtensorMap map_b, const RingParams p)
{
    qmv_ring_body<BITS, GS, SBP, V>(&map_w, &map_s, &map_b, p);
}

// The one-vector kernel: kOneWarps warps, kOneCtasPerSm CTAs per SM.
constexpr int kOneWarps = 12;
constexpr int kOneCtasPerSm = 1;
template <int BITS, int GS, bool SBP>
__global__ void __launch_bounds__(kOneWarps * 32, kOneCtasPerSm) qmv_one(const Params p)
{
    qmv_one_body<BITS, GS, SBP>(p);
}

template <int BITS, int GS, int V, bool SBP>
__global__ void __launch_bounds__(kThreadsVN, 1) qmv_streamed(const Params p)
{
    qmv_direct_body<BITS, GS, V, SBP>(p);
}

// The streamed kernel's x staging, once per call (kStageThreads a block).
constexpr int kStageThreads = 128;
template <int BITS>
__global__ void __launch_bounds__(kStageThreads)
    qmv_stage_x(const uint16_t *x, int K, int S_row, int V, uint8_t *out, unsigned *counters, int ncounters)
{
    stage_all_body<BITS>(x, K, S_row, V, out, counters, ncounters);
}

}  // namespace qmv
