// Problem geometry shared by the host launcher and the kernels.
//
// The K-split count and every split boundary are functions of (K, bits,
// group_size) alone. They fix the fp32 summation order of each output, so
// they must never depend on M: that is what keeps column j of an M-vector
// call bit-identical to an M = 1 call on the same vector (mlxcel issue #1289,
// "The observation this rests on").
#pragma once

#include <cstdint>

namespace qmv {

constexpr int kWarps = 8;                      // warps per CTA
constexpr int kThreads = kWarps * 32;          // 256
constexpr int kRowsPerWarp = 8;                // one TMA box is 8 rows tall
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;  // 64
constexpr int kSlices = 8;                     // lanes sharing a row pair; one group each per stage
constexpr int kBoxBytes = 128;                 // TMA box inner extent (bytes) = 128B swizzle span
constexpr int kBoxSmem = kBoxBytes * kRowsPerWarp;  // 1024 bytes per box in shared memory
constexpr int kRingBytesPerWarp = 8192;        // weight tiles in flight per warp
constexpr int kMaxSplitElems = 2048;           // K elements per split, at most
constexpr int kMaxM = 16;
constexpr int kMaxChunksPerCta = 64;           // a CTA that takes all of K holds at most this many chunks

__host__ __device__ constexpr int group_bytes(int bits, int gs) { return gs * bits / 8; }
__host__ __device__ constexpr int groups_per_box(int bits, int gs) { return kBoxBytes / group_bytes(bits, gs); }
__host__ __device__ constexpr int boxes_per_stage(int bits, int gs)
{
    return kSlices * group_bytes(bits, gs) / kBoxBytes;
}
__host__ __device__ constexpr int stage_bytes(int bits, int gs) { return boxes_per_stage(bits, gs) * kBoxSmem; }
__host__ __device__ constexpr int ring_stages(int bits, int gs) { return kRingBytesPerWarp / stage_bytes(bits, gs); }
__host__ __device__ constexpr int x_stride(int gs) { return gs + 4; }  // floats per group, padded

// Number of 128-byte weight boxes along one row (the last may be partial).
inline int row_boxes(int K, int bits, int gs)
{
    const int G = K / gs;
    const int gpb = groups_per_box(bits, gs);
    return (G + gpb - 1) / gpb;
}

// K-split count: the fewest splits that keep each split within kMaxSplitElems,
// raised to the next divisor of the box count (equal splits) when one exists
// below twice that minimum.
inline int split_count(int K, int bits, int gs)
{
    const int nbox = row_boxes(K, bits, gs);
    int max_boxes = (kMaxSplitElems / gs) / groups_per_box(bits, gs);
    if (max_boxes < 1) max_boxes = 1;
    const int ks_min = (nbox + max_boxes - 1) / max_boxes;
    for (int ks = ks_min; ks <= 2 * ks_min && ks <= nbox; ++ks)
        if (nbox % ks == 0) return ks;
    return ks_min;
}

// Split s covers boxes [s*nbox/ks, (s+1)*nbox/ks) of every row.
__host__ __device__ inline int split_box_begin(int s, int nbox, int ks)
{
    return int((long long)s * nbox / ks);
}

// Most groups any split holds (sizes the activation staging buffer).
inline int max_split_groups(int K, int bits, int gs)
{
    const int nbox = row_boxes(K, bits, gs), ks = split_count(K, bits, gs);
    const int gpb = groups_per_box(bits, gs), G = K / gs;
    int best = 0;
    for (int s = 0; s < ks; ++s) {
        int g0 = split_box_begin(s, nbox, ks) * gpb;
        int g1 = split_box_begin(s + 1, nbox, ks) * gpb;
        if (g1 > G) g1 = G;
        if (g1 - g0 > best) best = g1 - g0;
    }
    return best;
}

struct SmemLayout {
    int ring, xs, sx, bar, total;  // byte offsets from the 1024-aligned base, and the size to request
};

// gsm: the most groups of x one CTA stages (all of K, or one chunk).
__host__ __device__ inline SmemLayout smem_layout(int bits, int gs, int V, int gsm)
{
    SmemLayout L;
    L.ring = 0;
    L.xs = kWarps * kRingBytesPerWarp;
    L.sx = L.xs + V * gsm * x_stride(gs) * 4;
    L.bar = (L.sx + V * gsm * 4 + 15) & ~15;
    const int end = L.bar + kWarps * ring_stages(bits, gs) * 8;
    L.total = end + 1024;  // slack for aligning the dynamic base to 1024 bytes
    return L;
}

// Kernel arguments other than the weight tensor map.
//
// K is cut into `ks` chunks (the splits above). The chunks fix the order of
// the fp32 sum; how they are shared out is free: a CTA processes the chunks
// [blockIdx.y * cps, blockIdx.y * cps + cps), with cps = ks (one CTA sees all
// of K and folds the chunk values in registers) or cps = 1 (one chunk per
// CTA; the chunk values meet in the workspace and the CTA that finishes a row
// tile last folds them). Both give the same bits.
struct Params {
    const uint16_t *scales;   // bf16 bits [N, G]
    const uint16_t *biases;   // bf16 bits [N, G]
    const uint16_t *x;        // bf16 bits [V, K]
    void *y;                  // bf16 bits or float [V, N]
    float *partials;          // [ks, V, N] when cps < ks
    unsigned *counters;       // [ntiles] when cps < ks, zero between calls
    unsigned *err;            // device error word
    int N, K, G, ks, nbox, cps, gsm, ntiles, f32_out;
};

}  // namespace qmv
