// Problem geometry shared by the host launcher and the kernels.
//
// The fp32 summation order of an output is fixed by K alone (64-element
// subgroups, 2048-element chunks). It never depends on M, on the CTA shape or
// on the GPU: that is what keeps column j of an M-vector call bit-identical to
// an M = 1 call on the same vector (mlxcel issue #1289, "The observation this
// rests on").
#pragma once

#include <cstdint>

namespace qmv {

constexpr int kSub = 64;            // elements per subgroup: one lane's share of a chunk row
constexpr int kChunkSubs = 32;      // subgroups per chunk, one per lane of a warp
constexpr int kChunkElems = kSub * kChunkSubs;
constexpr int kRows = 4;            // rows per work unit; every lane of the warp works on all of them
constexpr int kMaxM = 16;
constexpr int kXsB16 = 144;         // bytes per staged subgroup, one-vector kernel: 128 B of bf16 x'' + 16 B of (sx, f1, f2, 0)
constexpr int kXsF32 = 272;         // bytes per staged subgroup and vector, streamed kernel: 256 B of fp32 x' + (sx, f1, f2, 0)

__host__ __device__ constexpr int sub_bytes(int bits) { return kSub * bits / 8; }
__host__ __device__ constexpr int chunk_bytes(int bits) { return kChunkElems * bits / 8; }
__host__ __device__ inline int subs_per_row(int K) { return K / kSub; }
// Number of K-chunks of a row (the last one may hold fewer than 32 subgroups).
__host__ __device__ inline int chunk_count(int K) { return (subs_per_row(K) + kChunkSubs - 1) / kChunkSubs; }

// Arguments common to both kernels.
//
// CTA (i, j) owns the row blocks [i*NB/grid_rows, (i+1)*NB/grid_rows) (4 rows
// each) and the chunks [j*cpc, min((j+1)*cpc, ks)). Chunk values meet in
// shared memory; with cpc = ks the CTA folds them into y, otherwise they go
// through the workspace and the CTA that completes a row range last folds all
// ks of them.
struct Params {
    const uint8_t *w;         // packed weights [N, row_bytes]
    const uint16_t *scales;   // bf16 bits [N, G]
    const uint16_t *biases;   // bf16 bits [N, G]
    const uint16_t *x;        // bf16 bits [V, K]
    void *y;                  // bf16 bits or float [V, N]
    float *partials;          // [ks, V, N] when cpc < ks
    unsigned *counters;       // [NB] (one per first row block of a range) when cpc < ks; zero between calls
    unsigned *err;            // device error word
    int N, K, G;              // G = K / group_size
    int S_row;                // subgroups per row
    int ks;                   // chunks per row
    int row_bytes;
    int NB;                   // row blocks of the matrix
    int grid_rows;            // CTAs along the rows
    int cpc;                  // chunks per CTA
    int max_rb;               // row blocks of the largest CTA share
    int f32_out;
    const uint8_t *xs_staged; // streamed kernel: the call's staged cells [V][S_row] (qmv_stage_x)
    int sb_packed;            // 1: scales is the interleaved uint32 array (scale low, bias high), biases unused
    int early_weights;        // one-vector kernels: 1 = weights, scales, biases may be read before the wait for
                              // the preceding grid (QMV_PDL); 0 = nothing is read before that wait
};

// The one-vector kernel's ring: units are (row block, piece) pairs, a piece
// being uc consecutive chunks of the CTA's range; producer warps stream them
// through `slots` shared-memory slots (weights, then the scale and bias
// boxes) and the consumer warps take them in order from a shared counter.
// How a unit's weights travel:
constexpr int kUnitPieces = 0;  // one bulk copy per row; scale/bias boxes per row (1-D maps)
constexpr int kUnitRows = 1;    // whole rows: the 4 rows are contiguous, one bulk copy
constexpr int kUnitTiles = 2;   // one 2-D box of 4 rows x pitch bytes; one 2-D scale and one bias box
struct RingParams : Params {
    int uc;                   // chunks per unit
    int unit_mode;            // kUnitPieces, kUnitRows or kUnitTiles
    int pitch;                // bytes per unit row in a slot
    int sb_mode_unit;         // 1: one scale box and one bias box per unit; 0: one of each per row
    int sbox;                 // elements per metadata box (a multiple of 16 bytes; tiles: 4 rows of uc chunks' groups)
    int slots;                // ring slots (a multiple of the producer warps)
    int consumers;            // consumer warps; warps consumers.. are producers
};

__host__ __device__ inline int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Vectors per pass of the streamed kernel (two passes above eight).
__host__ __device__ constexpr int vectors_per_pass(int V) { return V <= 8 ? V : (V + 1) / 2; }

// Shared memory of the streamed kernel, as byte offsets from a 128-aligned
// base: staged x, chunk values, and (two passes) each warp's unit of weights
// (4 rows x 32 lanes x one subgroup).
struct SmemLayout {
    int xs, cv, wbuf, misc, total;
};

__host__ __device__ inline SmemLayout smem_layout(int bits, int V, int warps, int nsub, int max_rb, int cpc)
{
    SmemLayout L;
    L.xs = 0;
    L.cv = align_up(V * nsub * kXsF32, 16);
    L.wbuf = align_up(L.cv + max_rb * kRows * cpc * V * 4, 16);
    L.misc = L.wbuf + (vectors_per_pass(V) < V ? warps * kRows * 32 * sub_bytes(bits) : 0);
    L.total = L.misc + 16 + 128;  // next-unit counter and the x barrier; slack for aligning the dynamic base
    return L;
}

// Shared memory of the one-vector kernel qmv_one, as byte offsets from a
// 128-aligned base: staged x'' cells (kXsB16 bytes a subgroup: 128 bytes of
// x'' and its (sx, f1, f2, 0)), chunk values.
struct OneLayout {
    int xs, cv, total;
};

__host__ __device__ inline OneLayout one_layout(int nsub, int max_rb, int cpc)
{
    OneLayout L;
    L.xs = 0;
    L.cv = align_up(nsub * kXsB16, 16);
    L.total = L.cv + max_rb * kRows * cpc * 4 + 128;  // slack for aligning the dynamic base
    return L;
}

// Shared memory of the one-vector ring kernel, as byte offsets from a
// 128-aligned base: the ring, the raw x (128 bytes a subgroup, landed by one
// bulk copy), the staged x'' cells (kXsB16 bytes a subgroup), chunk values,
// the slot barriers and the x barrier, counters.
constexpr int kBoxAlign = 128;  // shared-memory alignment of a tensor-map box
struct RingLayout {
    int slot_bytes, sb_off, sbs;  // slot size, offset of the scale/bias boxes in a slot, bytes per box
    int ring, xr, xc, cv, bar, misc, total;
};

// Metadata element bytes: a bf16 scale or bias, or an interleaved pair.
__host__ __device__ constexpr int sb_elem_bytes(int sb_packed) { return sb_packed ? 4 : 2; }

__host__ __device__ inline RingLayout ring_layout(int pitch, int sb_mode_unit, int sbox, int sb_packed, int slots,
                                                  int nsub, int max_rb, int cpc, int V = 1)
{
    RingLayout L;
    L.sbs = align_up(sbox * sb_elem_bytes(sb_packed), kBoxAlign);
    L.sb_off = align_up(kRows * pitch, kBoxAlign);
    // boxes per slot: one per unit or one per row, of each metadata tensor
    L.slot_bytes = L.sb_off + (sb_mode_unit ? 1 : kRows) * (sb_packed ? 1 : 2) * L.sbs;
    L.ring = 0;
    L.xr = slots * L.slot_bytes;
    L.xc = L.xr + (V == 1 ? nsub * 128 : 0);
    L.cv = align_up(L.xc + (V == 1 ? nsub * kXsB16 : V * nsub * kXsF32), 16);
    L.bar = align_up(L.cv + max_rb * kRows * cpc * V * 4, 16);
    L.misc = L.bar + (2 * slots + 1) * 8;
    L.total = L.misc + 32 + kBoxAlign;  // next-unit counter, abort flag, issued counts; alignment slack
    return L;
}

}  // namespace qmv
