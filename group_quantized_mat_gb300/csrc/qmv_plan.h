// Problem geometry shared by the host launcher and the kernels.
//
// The fp32 summation order of an output is fixed by the group size and the
// K-chunks below, which depend on K and group_size alone. They never depend on
// M, on the CTA shape or on the GPU: that is what keeps column j of an
// M-vector call bit-identical to an M = 1 call on the same vector (mlxcel
// issue #1289, "The observation this rests on").
#pragma once

#include <cstdint>

namespace qmv {

constexpr int kSlices = 8;          // lanes sharing a row; slice j takes groups j, j+8, ... of a chunk
constexpr int kChunkElems = 2048;   // K elements per chunk (the last chunk of a row may be shorter)
constexpr int kBoxBytes = 128;      // TMA box inner extent = 128B swizzle span
constexpr int kMaxM = 16;
constexpr int kMaxWarps = 16;       // warps per CTA
constexpr int kMaxChunksPerCta = 64;

__host__ __device__ constexpr int group_bytes(int bits, int gs) { return gs * bits / 8; }
__host__ __device__ constexpr int groups_per_box(int bits, int gs) { return kBoxBytes / group_bytes(bits, gs); }
__host__ __device__ constexpr int boxes_per_stage(int bits, int gs) { return kSlices * group_bytes(bits, gs) / kBoxBytes; }
__host__ __device__ constexpr int chunk_groups(int gs) { return kChunkElems / gs; }  // a multiple of kSlices
__host__ __device__ constexpr int x_stride(int gs) { return gs + 4; }               // floats per staged group

// Number of K-chunks of a row: ceil(G / chunk_groups).
__host__ __device__ inline int chunk_count(int K, int gs)
{
    const int G = K / gs;
    return (G + chunk_groups(gs) - 1) / chunk_groups(gs);
}

// Kernel arguments other than the weight tensor map.
//
// A CTA owns up to RB row blocks (4R rows each) and the chunks
// [blockIdx.y * cps, blockIdx.y * cps + cps). Its work units are (row block,
// chunk phase) pairs, a chunk phase being one of H contiguous blocks of the
// CTA's chunks; warp w processes units w, w + warps, ... Chunk values meet in
// shared memory; with cps = ks the CTA folds them into y, otherwise they go
// through the workspace and the CTA that completes a row tile last folds all
// ks of them.
struct Params {
    const uint16_t *scales;   // bf16 bits [N, G]
    const uint16_t *biases;   // bf16 bits [N, G]
    const uint16_t *x;        // bf16 bits [V, K]
    void *y;                  // bf16 bits or float [V, N]
    float *partials;          // [ks, V, N] when cps < ks
    unsigned *counters;       // [ntiles] when cps < ks, zero between calls
    unsigned *err;            // device error word
    int N, K, G;
    int ks;                   // chunks per row
    int cps;                  // chunks per CTA: ks or 1
    int RB, H;                // row blocks (at most) and chunk phases per CTA
    int warps;                // warps per CTA; warp w takes units w, w + warps, ...
    int NB;                   // row blocks of the matrix (ceil(N / rows per block))
    int balanced;             // 1: CTA i takes row blocks [i*NB/grid, (i+1)*NB/grid)
    int stages;               // weight stages in flight per warp (a power of two)
    int gsm;                  // groups of x one CTA stages (its chunk range)
    int ntiles;               // row tiles (counters) when cps < ks
    int f32_out;
};

// Shared memory of one CTA, as byte offsets from a 1024-aligned base.
struct SmemLayout {
    int ring, xs, sx, cv, bar, total;
};

// rows_per_block = 4 * R; one stage = boxes_per_stage boxes of (128 B x rows_per_block).
__host__ __device__ inline int stage_bytes(int bits, int gs, int rows_per_block)
{
    return boxes_per_stage(bits, gs) * kBoxBytes * rows_per_block;
}

__host__ __device__ inline SmemLayout smem_layout(int bits, int gs, int V, int rows_per_block, int warps, int stages,
                                                  int gsm, int cps, int tile_rows)
{
    SmemLayout L;
    L.ring = 0;
    L.xs = warps * stages * stage_bytes(bits, gs, rows_per_block);
    L.sx = L.xs + V * gsm * x_stride(gs) * 4;
    L.cv = L.sx + V * gsm * 4;
    L.bar = (L.cv + cps * tile_rows * V * 4 + 15) & ~15;
    const int end = L.bar + warps * stages * 8;
    L.total = end + 1024;  // slack for aligning the dynamic base to 1024 bytes
    return L;
}

}  // namespace qmv
