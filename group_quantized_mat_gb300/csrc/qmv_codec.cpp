// Packed-weight codec of the affine group-quantized mat-vec library (host code).
//
// Field j of a uint32 word holds element (word * 32/bits + j) of its row at bit
// positions [bits*j, bits*j + bits): field 0 in the low bits. This is the layout
// read by the qdot masks of mlxcel issue #1289 ("Correction to the obvious
// sketch": element 4i <-> mask 0x000f, element 4i+1 <-> mask 0x00f0) and the
// "plain bit packing" of llama.cpp PR #159 ("How").
#include <cstdint>
#include <cstring>

#include "qmv.h"

namespace {

bool codec_args_ok(int64_t N, int64_t K, int bits)
{
    return (bits == 2 || bits == 4) && N >= 1 && K >= 1 && (K * bits) % 32 == 0 &&
           N <= (int64_t(1) << 40) / K;
}

}  // namespace

extern "C" size_t qmv_packed_words(int64_t N, int64_t K, int bits)
{
    if (!codec_args_ok(N, K, bits)) return 0;
    return size_t(N) * size_t(K * bits / 32);
}

extern "C" qmv_status qmv_pack(const uint8_t *q, uint32_t *w_q, int64_t N, int64_t K, int bits)
{
    if (!q || !w_q) return QMV_ERR_NULL;
    if (bits != 2 && bits != 4) return QMV_ERR_BITS;
    if (!codec_args_ok(N, K, bits)) return QMV_ERR_SHAPE;
    const int per_word = 32 / bits;
    const uint32_t limit = 1u << bits;
    const int64_t words = N * K / per_word;
    // Rows are contiguous in both arrays, so the matrix packs as one stream.
    for (int64_t wi = 0; wi < words; ++wi) {
        const uint8_t *src = q + wi * per_word;
        uint32_t word = 0;
        for (int j = 0; j < per_word; ++j) {
            const uint32_t v = src[j];
            if (v >= limit) return QMV_ERR_VALUE;
            word |= v << (bits * j);
        }
        w_q[wi] = word;
    }
    return QMV_OK;
}

extern "C" qmv_status qmv_pack_sb(const uint16_t *scales, const uint16_t *biases, uint32_t *sb, int64_t N, int64_t G)
{
    if (!scales || !biases || !sb) return QMV_ERR_NULL;
    if (N < 1 || G < 1 || N > (int64_t(1) << 40) / G) return QMV_ERR_SHAPE;
    const int64_t n = N * G;
    for (int64_t i = 0; i < n; ++i) sb[i] = uint32_t(scales[i]) | (uint32_t(biases[i]) << 16);
    return QMV_OK;
}

extern "C" qmv_status qmv_unpack(const uint32_t *w_q, uint8_t *q, int64_t N, int64_t K, int bits)
{
    if (!q || !w_q) return QMV_ERR_NULL;
    if (bits != 2 && bits != 4) return QMV_ERR_BITS;
    if (!codec_args_ok(N, K, bits)) return QMV_ERR_SHAPE;
    const int per_word = 32 / bits;
    const uint32_t mask = (1u << bits) - 1u;
    const int64_t words = N * K / per_word;
    for (int64_t wi = 0; wi < words; ++wi) {
        const uint32_t word = w_q[wi];
        uint8_t *dst = q + wi * per_word;
        for (int j = 0; j < per_word; ++j) dst[j] = uint8_t((word >> (bits * j)) & mask);
    }
    return QMV_OK;
}
