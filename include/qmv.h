/*
 * qmv.h -- C ABI of the GB300 (sm_103a) group-quantized mat-vec library: the
 * affine mode below, and the mxfp4 mode (qmv_mxfp4_run).
 *
 *   y[m, n] = sum_i ( s[n, i/gs] * q[n, i] + b[n, i/gs] ) * x[m, i]
 *
 * for M activation vectors x[M, K] (bf16), N output rows, packed b-bit weights
 * q (bits = 4 or 2), one bf16 scale s and one bf16 bias b per group of gs = 64
 * or 128 consecutive weights along K, bf16 output y[M, N].
 *
 * Source of the operation (group_quantized_mat pages):
 *  - mlxcel issue #1289 "perf(metal): an order-preserving streamed qmv ...":
 *    section "Correction to the obvious sketch: qdot does not dequantize"
 *    (the affine form scale*q + bias, the factored group dot
 *    scale*sum(q*x) + bias*sum(x), the field masks of a packed word);
 *    sections "The observation this rests on" and "Step 2" (one weight read
 *    serving M streamed vectors, each result bit-identical to the M = 1 run).
 *  - llama.cpp PR #159 "metal: PQ2_0 and Q2_0 mat-vec dot in exact float",
 *    section "How" (2-bit fields, field 0 in the low bits; group sizes 64
 *    and 128).
 *  - mlxcel PR #1681 "perf(cuda/quant): block output rows per warp ...",
 *    section "Not covered" (scale and bias applied once per group).
 *
 * Every function here is host code. Pointers documented as "device" must be
 * device (or managed) memory of the current CUDA device; "host" pointers are
 * ordinary host memory. The library never takes ownership of a caller's
 * buffer and never frees one.
 */
#ifndef QMV_H
#define QMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the shared library (it is built with hidden default visibility). */
#if defined(__GNUC__)
#define QMV_API __attribute__((visibility("default")))
#else
#define QMV_API
#endif

/* Return codes. Every entry point validates its arguments on the host before
 * touching the GPU and returns a code instead of launching on bad input. */
typedef enum qmv_status {
    QMV_OK = 0,
    QMV_ERR_NULL = 1,       /* a required pointer is NULL                                  */
    QMV_ERR_BITS = 2,       /* bits is not 2 or 4                                          */
    QMV_ERR_GROUP = 3,      /* group_size is not 64 or 128                                 */
    QMV_ERR_SHAPE = 4,      /* N < 1, K < 1, K % group_size != 0, or a size overflows
                               (N > 2^30, K > 2^24, N * K / group_size >= 2^31)          */
    QMV_ERR_M_RANGE = 5,    /* M is not in [1, QMV_MAX_M]                                  */
    QMV_ERR_ALIGN = 6,      /* w_q, x, scales, biases or workspace not 16-byte aligned;
                               y not 2-byte aligned (4 for an fp32 y)                     */
    QMV_ERR_CUDA = 7,       /* a CUDA runtime call failed (launch, device query, encode)   */
    QMV_ERR_WORKSPACE = 8,  /* workspace is smaller than qmv_workspace_size()              */
    QMV_ERR_VALUE = 9,      /* qmv_pack: an input value does not fit in `bits` bits        */
    QMV_ERR_FLAGS = 10      /* unknown bits set in `flags`                                 */
} qmv_status;

/* The CUDA stream type (identical to cudaStream_t; 0 is the legacy default stream). */
typedef struct CUstream_st *qmv_stream_t;

/* Widest activation batch one launch serves from a single read of the weights
 * (the speculative-verify width). */
#define QMV_TILE_M 16

/* Most vectors per call. A call with M > QMV_TILE_M runs as consecutive
 * launches of QMV_TILE_M vectors and one of the remainder, reading the weights
 * once per launch; every column's arithmetic is the same as at M = 1. (Above
 * the batch limit the pages hand off to a dense quantized mat-mat, issue #1289
 * "Scope limits"; this tiling is the order-preserving stand-in.) */
#define QMV_MAX_M 256

/* ------------------------------------------------------------------ codec */

/* Number of uint32 words of the packed weight matrix: N * K * bits / 32.
 * Returns 0 for invalid arguments (bits not in {2,4}, N < 1, K < 1, or K * bits
 * not a multiple of 32). */
QMV_API size_t qmv_packed_words(int64_t N, int64_t K, int bits);

/* Packs q[N, K] (host, row-major uint8, each value < 2^bits) into
 * w_q[N, K*bits/32] (host, row-major uint32, caller-allocated). Field j of a
 * word holds element (word_index * 32/bits + j) of the row at bit positions
 * [bits*j, bits*j + bits): field 0 in the low bits, little-endian
 * (issue #1289 "Correction..."; PR #159 "How").
 * Errors: QMV_ERR_NULL, QMV_ERR_BITS, QMV_ERR_SHAPE (K*bits % 32 != 0),
 * QMV_ERR_VALUE (a value >= 2^bits; w_q is then left unspecified). */
QMV_API qmv_status qmv_pack(const uint8_t *q, uint32_t *w_q, int64_t N, int64_t K, int bits);

/* Inverse of qmv_pack (host to host). Same errors except QMV_ERR_VALUE. */
QMV_API qmv_status qmv_unpack(const uint32_t *w_q, uint8_t *q, int64_t N, int64_t K, int bits);

/* Interleaves the per-group metadata into one word per group (host to host):
 * sb[i] = scales[i] | (biases[i] << 16) for i < N*G, scales and biases being
 * bf16 bit patterns [N, G], sb uint32 [N, G] (caller-allocated). A call with
 * QMV_SB_INTERLEAVED reads this array through its `scales` argument: one load
 * (or one tensor-map box) brings both values of a group where the separate
 * arrays need two (PR #1681 "What is here as an instrument" prices the scale
 * and bias loads). The arithmetic, and so every result, is unchanged.
 * Errors: QMV_ERR_NULL, QMV_ERR_SHAPE (N < 1, G < 1 or N*G >= 2^40). */
QMV_API qmv_status qmv_pack_sb(const uint16_t *scales, const uint16_t *biases, uint32_t *sb, int64_t N, int64_t G);

/* ------------------------------------------------------------------- plan */

/* Number of K-chunks (2048 elements each, the last one possibly shorter) that
 * fix the fp32 summation order of a (N, K, bits, group_size) problem, or 0 for
 * invalid arguments. It depends on K only -- never on M -- so the order of
 * every output is the same for every M (the basis of the bit-identity
 * guarantee below). */
QMV_API int qmv_split_count(int N, int K, int bits, int group_size);

/* Bytes of device workspace a call with these arguments needs: for M >= 2 the
 * call's staged activations (M x K/64 cells of 144 or 272 bytes), plus, when
 * CTAs split K, one counter per 4-row block and the per-chunk partial sums
 * (0 for M = 1 when one CTA covers all K-chunks of its rows). Returns 0 for
 * invalid arguments too. */
QMV_API size_t qmv_workspace_size(int M, int N, int K, int bits, int group_size);

/* ------------------------------------------------------------------- run */

/* y = W . x for M vectors, asynchronously on `stream`.
 *
 *  w_q     device, uint32 [N, K*bits/32] from qmv_pack, 16-byte aligned.
 *  scales  device, bf16 bit patterns [N, K/group_size], row-major, 16-byte aligned.
 *  biases  device, bf16 bit patterns [N, K/group_size], row-major, 16-byte aligned.
 *  x       device, bf16 [M, K], row-major (vector-major), 16-byte aligned.
 *  y       device, bf16 [M, N], row-major; must not overlap any input.
 *  M       1 .. QMV_MAX_M.  N, K >= 1; K a multiple of group_size.
 *  bits    4 or 2.  group_size 64 or 128.
 *
 * Arithmetic: fp32. Each group is evaluated in the factored form
 * s * (sum q x) + b * (sum x) (no dequantized weight is formed), then rounded
 * once to bf16 (nearest even). The fp32 operation order for an output element
 * depends only on (N, K, bits, group_size) and the element's row: column j of
 * an M-vector call is bit-identical to an M = 1 call on x[j] (issue #1289
 * "The observation this rests on": identity that follows from the arithmetic
 * itself, not from a tolerance).
 *
 * The call returns after enqueueing. Most calls need no scratch (M = 1 with
 * the whole of K per CTA); M >= 2, and problems whose CTAs split K, need a
 * workspace (qmv_workspace_size). qmv_run then uses one owned by the library,
 * one per device, kept until exit. The first call that needs more than the
 * current one allocates it with cudaMalloc (after cudaFree of the smaller one,
 * which waits for the device's work in flight): that call is not stream-ordered,
 * may block the host until the device is idle, and must not be made during
 * stream capture. No other qmv_run call allocates or synchronizes. Every call
 * on a device shares the one library workspace, so qmv_run calls that overlap
 * on the GPU (issued to different streams, or from concurrent host threads)
 * race on it and give undefined results: concurrent callers use qmv_run_ex
 * with one workspace each, or serialize their calls on one stream.
 *
 * Errors: QMV_ERR_NULL, QMV_ERR_BITS, QMV_ERR_GROUP, QMV_ERR_SHAPE,
 * QMV_ERR_M_RANGE, QMV_ERR_ALIGN (host checks, nothing launched);
 * QMV_ERR_CUDA when the workspace allocation, the tensor-map encode or the
 * launch fails (cudaGetLastError is consumed). */
QMV_API qmv_status qmv_run(const uint32_t *w_q, const uint16_t *scales, const uint16_t *biases,
                   const uint16_t *x, uint16_t *y, int M, int N, int K, int bits,
                   int group_size, qmv_stream_t stream);

/* Flags for qmv_run_ex. */
#define QMV_F32_OUT 0x1u             /* y is float [M, N]: the fp32 value before bf16 rounding */
#define QMV_FORCE_M1_PER_COLUMN 0x2u /* serve the M vectors as M separate M = 1 launches       */
/* Launch with a programmatic dependency on the preceding kernel of the stream:
 * the call may start streaming w_q, scales and biases before that kernel has
 * finished (x, y and the workspace are touched only after it has). Set it only
 * when the preceding kernel does not write w_q, scales or biases -- the
 * decode-loop case, where weights are constant. (Without the flag a one-vector
 * launch that needs no scratch still carries a programmatic dependency, so that
 * its set-up overlaps the preceding kernel's tail, but it reads and writes
 * nothing before that kernel has completed: stream order is unchanged.) */
#define QMV_PDL 0x4u
/* `scales` is the uint32 [N, K/group_size] array of qmv_pack_sb (16-byte
 * aligned); `biases` is not read and may be NULL. */
#define QMV_SB_INTERLEAVED 0x8u

/* qmv_run with an explicit workspace and flags.
 *
 *  workspace        device, 16-byte aligned, at least qmv_workspace_size(M, N, K,
 *                   bits, group_size) bytes, or NULL to use the library workspace.
 *                   Scratch only: a call needs no particular contents (it clears
 *                   what must start at zero on `stream` itself) and leaves
 *                   unspecified ones, so one workspace serves any sequence of
 *                   problem shapes. Calls sharing one workspace must not overlap
 *                   on the GPU.
 *  workspace_bytes  its size in bytes (ignored when workspace is NULL).
 *  flags            bitwise OR of QMV_* flags above.
 * Additional errors: QMV_ERR_WORKSPACE, QMV_ERR_FLAGS. */
QMV_API qmv_status qmv_run_ex(const uint32_t *w_q, const uint16_t *scales, const uint16_t *biases,
                      const uint16_t *x, void *y, int M, int N, int K, int bits,
                      int group_size, void *workspace, size_t workspace_bytes,
                      unsigned flags, qmv_stream_t stream);

/* Size of the fixed scratch array behind qmv_run_noalloc (8 MiB per device). */
#define QMV_NOALLOC_SCRATCH_BYTES (8u << 20)

/* qmv_run without any device allocation. The paper has no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc -- engines whose
 * device memory all belongs to their own pool allocator, and latency-bound
 * decode loops where cudaMalloc's implicit device synchronization is not
 * acceptable. qmv_run allocates its workspace on first use and qmv_run_ex
 * needs a caller-allocated one; this call needs neither.
 *
 * Arguments, layouts, results (bit for bit) and the host-side errors are those
 * of qmv_run. The scratch that K-split problems need comes from one static
 * device array of QMV_NOALLOC_SCRATCH_BYTES that every GPU loading the library
 * holds until exit; no cudaMalloc, cudaFree or allocating library routine is
 * called. All calls on a device share the array, so
 * calls that overlap on the GPU (other streams, or concurrent host threads)
 * race and give undefined results.
 *
 * The first call on a device, whatever its shape, looks up the array's
 * device address (cudaGetSymbolAddress) with that device current, which may
 * load the library's device code and wait for the device; later calls on that
 * device make no such lookup.
 *
 * Errors: those of qmv_run, checked first and in the same order; then
 * QMV_ERR_WORKSPACE when the problem's qmv_workspace_size() exceeds
 * QMV_NOALLOC_SCRATCH_BYTES (nothing launched); QMV_ERR_CUDA when the address
 * lookup or a launch fails (qmv_last_cuda_error() says which). */
QMV_API qmv_status qmv_run_noalloc(const uint32_t *w_q, const uint16_t *scales, const uint16_t *biases,
                                   const uint16_t *x, uint16_t *y, int M, int N, int K, int bits,
                                   int group_size, qmv_stream_t stream);

/* ------------------------------------------------------------------ mxfp4 */

/* y = W . x in the mxfp4 mode, asynchronously on `stream`:
 *
 *   y[m, n] = sum_i 2^(e[n, i/32] - 127) * e2m1(q[n, i]) * x[m, i]
 *
 * The pages name an order-preserving streamed qmv for the fp quantization
 * modes ("mxfp4") as the second phase of the work (issue #1289, "Scope limits,
 * stated honestly") without giving the format; this is the OCP MX v1.0 MXFP4
 * format:
 *  - element: E2M1 code: sign (bit 3), exponent (bits 2..1, bias 1) and
 *    mantissa (bit 0). Exponent 0 is subnormal, so the values are
 *    +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *  - scale: one E8M0 byte e per 32 consecutive elements along K, 2^(e - 127);
 *    e = 255 is NaN.
 *
 *  w_q     device, uint32 [N, K/8], 16-byte aligned: the codes packed as 4-bit
 *          fields exactly as qmv_pack(q, w_q, N, K, 4) packs them (element 0
 *          in the low nibble), so each 32-block is one 16-byte vector.
 *  scales  device, uint8 [N, K/32], row-major (no alignment needed).
 *  x       device, bf16 [M, K], row-major, 16-byte aligned.
 *  y       device, bf16 [M, N] (fp32 with QMV_F32_OUT), row-major; no overlap
 *          with any input.
 *  M       1 .. QMV_MAX_M (launches of QMV_TILE_M vectors). N >= 1,
 *          K >= 32 and a multiple of 32.
 *  flags   QMV_F32_OUT and QMV_FORCE_M1_PER_COLUMN (as for qmv_run_ex).
 *
 * Arithmetic is fp32 in a fixed order that depends only on K and the
 * element's row, never on M:
 *  1. Each block of 32 forms two fma chains, over its even and its odd
 *     elements. The products are exact.
 *  2. The chain sums are added, then multiplied by the block's scale.
 *  3. Blocks b = l, l+32, l+64, ... are folded in order into partial l, for
 *     l = 0..31.
 *  4. The 32 partials are summed by a fixed xor tree.
 *  5. The result is rounded once to bf16.
 * So column j of an M-vector call is bit-identical to an M = 1 call on x[j].
 * No workspace and no device allocation: the call may be captured in a CUDA
 * graph.
 *
 * Errors:
 *  - QMV_ERR_NULL.
 *  - QMV_ERR_SHAPE: N < 1, K < 1, K % 32 != 0, N > 2^30, K > 2^24, or
 *    N * K/32 >= 2^31.
 *  - QMV_ERR_M_RANGE, QMV_ERR_ALIGN, QMV_ERR_FLAGS.
 *  - QMV_ERR_CUDA when a launch fails.
 * The host checks run before anything is launched. */
QMV_API qmv_status qmv_mxfp4_run(const uint32_t *w_q, const uint8_t *scales, const uint16_t *x, void *y,
                                 int M, int N, int K, unsigned flags, qmv_stream_t stream);

/* Zero-fills `bytes` of a caller workspace on `stream` (cudaMemsetAsync). Calls
 * do not need it (a workspace holds no state between calls); kept as a
 * convenience. */
QMV_API qmv_status qmv_workspace_init(void *workspace, size_t bytes, qmv_stream_t stream);

/* ------------------------------------------------------------ diagnostics */

/* Device-side error word of the current device: the one-vector kernel sets
 * bit 0 when a bounded wait for a weight tile ran out and bit 1 when a launch
 * shape breaks its shared-memory ring protocol (neither happens with the
 * library's own launch plans; the output of that launch is then invalid).
 * Synchronizes the device, stores the word in *word and clears it.
 * Errors: QMV_ERR_NULL, QMV_ERR_CUDA. */
QMV_API qmv_status qmv_device_error(unsigned *word);

/* Description of the last CUDA failure behind a QMV_ERR_CUDA returned to the
 * calling thread (the failing call, the CUDA error name and text). The string
 * is owned by the library and valid until the thread's next failing call. */
QMV_API const char *qmv_last_cuda_error(void);

/* Static, human-readable name of a status code. Never NULL. */
QMV_API const char *qmv_status_string(qmv_status status);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H */
