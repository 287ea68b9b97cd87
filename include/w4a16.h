/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) group-quantized INT4-weight x
 * bf16-activation matmul library.
 *
 *   y[M, N] = x[M, K] . dequant(W)[N, K]^T,   w[n][k] = (q[n][k] - z[n][k/G]) * scale[n][k/G]
 *
 * The dequantisation is the exact "(q - z) * scale" of the INT4 kernels in the
 * GRIMOIRE v1.7 release notes ("What changed"): q a 4-bit code, one bf16 scale
 * per (output row, K-group) with group G = 64 or 128, and z = 8 for the
 * symmetric GPTQ-Int4 checkpoints or a packed 4-bit zero point for the
 * asymmetric AutoRound W4A16 ones (same page, measurement table). The regimes
 * are those the same pages measure: one-row decode, 2-16 rows of batched
 * decode and speculative verify, the output-vocabulary head over all verify
 * rows in one pass, and 4,096-row prompts with the feed-forward gate fused in
 * (GRIMOIRE v1.8 release notes, "INT4 verify faster" and "INT4 prompt
 * processing").
 *
 * A third weight form, affine, rebuilds w[n][k] = scale[n][k/G] * q[n][k] +
 * bias[n][k/G] with a bf16 bias per group in place of the zero point: the MLX
 * affine 4-bit checkpoints that TensorFold PR #859 runs ("What this changes":
 * every code keeps its value, scale and bias; groups of 64). Its calls carry
 * "affine" in their names; the others take zero-point forms only.
 *
 * Canonical (input) layout, row-major, little-endian:
 *   qweight int32  [N][K/8]            nibble j (bits 4j..4j+3) of word c holds k = 8c + j
 *   scales  bf16   [N][K/G]            bf16 values passed as uint16_t bit patterns
 *   zeros   int32  [N][ceil(K/G/8)]    nibble j of word c holds the zero of group 8c + j
 *                                      (asymmetric only; unused nibbles ignored)
 *   biases  bf16   [N][K/G]            affine form only
 *
 * Conventions for every call:
 *   - Pointers named x, y, h, qweight, scales, zeros, packed, w_out are DEVICE
 *     pointers owned by the caller; the library allocates no device memory
 *     and keeps no pointer after a call returns.
 *   - Every compute call is asynchronous on `stream` (NULL = legacy default
 *     stream) and launches kernels on the calling thread's current device.
 *   - Return value: W4A16_OK (0) or a negative W4A16_ERR_* code. On any error
 *     detected before launch nothing is launched and no memory is written.
 *     W4A16_ERR_CUDA means a CUDA call failed; w4a16_last_cuda_error() gives
 *     its cudaError_t value (thread-local).
 *   - bf16 values are IEEE bfloat16 bit patterns in uint16_t; outputs are
 *     rounded to nearest-even from float32.
 *   - `sym` names the weight form: 0 = packed zero points, 1 = symmetric
 *     (z = 8; `zeros` is ignored and may be NULL), W4A16_AFFINE (2) =
 *     scale * q + bias, accepted only where a comment says so. Any other
 *     value is W4A16_ERR_INVALID_ARG (size queries return 0).
 *   - Supported sizes: 1 <= M, 1 <= N, 64 <= K, K % G == 0, G in {64, 128},
 *     M, N, K below 2^31 / 16.
 *   - Alignment: x, y, h 16 bytes; packed 256 bytes (cudaMalloc gives both).
 */
#ifndef W4A16_H_
#define W4A16_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without the CUDA headers (same type as the runtime's). */
typedef struct CUstream_st *w4a16_stream_t;

#define W4A16_OK 0
#define W4A16_ERR_INVALID_ARG (-1)  /* size, group, null pointer or reserved argument */
#define W4A16_ERR_MISALIGNED (-2)   /* a pointer breaks the alignment rules above */
#define W4A16_ERR_UNSUPPORTED (-3)  /* the current device is not an sm_103 GPU */
#define W4A16_ERR_CUDA (-4)         /* a CUDA call failed; see w4a16_last_cuda_error() */
#define W4A16_ERR_TIMEOUT (-5)      /* a bounded wait inside a kernel gave up */

/* Weight forms (the `sym` argument). */
#define W4A16_ZERO_POINTS 0
#define W4A16_SYMMETRIC 1
#define W4A16_AFFINE 2

/*
 * Size in bytes of the repacked weight that w4a16_repack (sym 0 or 1) or
 * w4a16_repack_affine (sym = W4A16_AFFINE) writes for an N x K weight (codes,
 * scales, and the zero points (sym = 0) or the biases (affine), each section
 * 256-byte aligned; rows padded to a multiple of 16). Returns 0 when the
 * sizes or the form are not supported.
 */
size_t w4a16_repacked_bytes(int N, int K, int group, int sym);

/*
 * Offline repack of one canonical weight (qweight, scales, zeros as above)
 * into the library's tiled layout in `packed` (w4a16_repacked_bytes bytes,
 * caller-allocated device memory). Pure bit moves: no value is rounded, so
 * every dequantised weight stays exactly (q - z) * scale. Rows are tiled 16 at
 * a time; within a tile and a 64-wide K chunk each of 32 lanes owns one
 * 16-byte run of codes for two rows and 16 consecutive k, the order in which
 * the kernels consume them. Scales (and zeros) sit per tile in blocks of four
 * groups. Padding rows get code 0, scale 0 and zero 0. Not timed on the hot
 * path; asynchronous on `stream`.
 */
int w4a16_repack(const int32_t *qweight, const uint16_t *scales, const int32_t *zeros,
                 int N, int K, int group, int sym, void *packed, w4a16_stream_t stream);

/* Size of the repacked gate/up pair of w4a16_repack_gateup or, for sym =
 * W4A16_AFFINE, w4a16_repack_affine_gateup (N_each rows each). */
size_t w4a16_gateup_repacked_bytes(int N_each, int K, int group, int sym);

/*
 * Offline repack of the feed-forward gate and up weights (two canonical
 * weights of N_each rows each) into one buffer whose 16-row tiles alternate
 * gate, up, gate, up, ... (N_each padded to a multiple of 128), so that one
 * tile of the prompt GEMM holds 128 gate rows and the 128 matching up rows.
 * The result is also a valid w4a16_repack buffer of 2 * round_up(N_each, 128)
 * rows in that interleaved order.
 */
int w4a16_repack_gateup(const int32_t *qw_gate, const uint16_t *sc_gate, const int32_t *z_gate,
                        const int32_t *qw_up, const uint16_t *sc_up, const int32_t *z_up,
                        int N_each, int K, int group, int sym, void *packed,
                        w4a16_stream_t stream);

/*
 * y[M][N] (bf16, row-major) = x[M][K] (bf16, row-major) . dequant(W)^T, with
 * W given as the output of w4a16_repack for the same (N, K, group, sym).
 * float32 accumulation; each group's partial sum is scaled in float32.
 * `scales` and `zeros` are reserved: scales and zero points travel inside
 * `packed`, and both must be NULL (else W4A16_ERR_INVALID_ARG).
 * Kernel choice: M <= 32 -> a decode kernel (each weight read and unpacked
 * once for all rows, multiply-adds on the tensor core): the one that stages x
 * once per CTA when M <= 8 and its grid fills the GPU, or for 9-16 rows of a
 * zero-point weight whose grid spans 1.5 CTAs per SM, else the one with a
 * weight ring per warp; M > 32 -> the tcgen05 GEMM. A CUDA-core one-row GEMV
 * is selectable (w4a16_set_kernel_override).
 * Results are bitwise reproducible run to run (no atomics in any sum).
 */
int w4a16_gemm(const uint16_t *x, const void *packed, const uint16_t *scales,
               const int32_t *zeros, int M, int N, int K, int group, int sym, uint16_t *y,
               w4a16_stream_t stream);

/*
 * Greedy pick over the output columns: argmax[m] = the first n at which the
 * bf16 output y[m][n] of w4a16_gemm (same x, packed, sizes) is largest, as
 * torch.argmax over a bf16 row returns it: among equal values the lowest n;
 * -0 equals +0; a NaN counts as the maximum. For the output-vocabulary head
 * this replaces reading back M x N logits with M indices (the GPU argmax
 * after the tall head in lucebox PR #823; one pass over all verify rows as in
 * the GRIMOIRE v1.8 release notes, "INT4 verify faster").
 *
 *   argmax  int64 [M], device, 8-byte aligned; written by this call
 *   y       bf16 [M][N] or NULL. M <= 32: the decode kernel forms the argmax
 *           in its epilogue and stores y only when y is not NULL (the logits
 *           need not exist). M > 32: required; the tcgen05 GEMM writes y and
 *           a second kernel reads it back.
 *
 * Launches three kernels on `stream` (zero the keys, the GEMM, turn keys
 * into indices), all taking part in programmatic overlap when it is on; the
 * result is ready when the stream reaches the end of the call. Errors as
 * w4a16_gemm.
 */
int w4a16_gemm_argmax(const uint16_t *x, const void *packed, int M, int N, int K, int group, int sym,
                      uint16_t *y, int64_t *argmax, w4a16_stream_t stream);

/*
 * Top-k of bf16 rows: the greedy pick on the GPU (lucebox PR #823,
 * description) widened to the k largest entries of each row of the logits
 * y [M][N], with the argmax's rules: largest value first; equal values
 * lowest column first (-0 equals +0); a NaN ranks above +inf (NaNs among
 * themselves by column). k = 1 gives w4a16_gemm_argmax's index.
 *
 *   y     bf16 [M][N], device, 2-byte aligned (16-byte aligned rows with N a
 *         multiple of 8 take 16-byte loads); read only
 *   k     1 <= k <= min(N, 1024)
 *   idx   int64 [M][k], device, 8-byte aligned: the columns, best first
 *   vals  bf16 [M][k], device, or NULL: y at those columns (bit patterns)
 *
 * One kernel on `stream`: per row, one cluster of up to 16 CTAs (two radix
 * passes of 8 bits over the order-preserving 16-bit codes of the values,
 * histograms summed over distributed shared memory, then a sort of the k
 * picks); it allocates nothing and takes part in programmatic overlap when
 * that is on. Errors: W4A16_ERR_INVALID_ARG (null y or idx, M or N out of
 * range, k out of range), W4A16_ERR_MISALIGNED, as w4a16_gemm otherwise.
 */
int w4a16_topk(const uint16_t *y, int M, int N, int k, int64_t *idx, uint16_t *vals, w4a16_stream_t stream);

/*
 * w4a16_gemm into y (required: the logits the selection reads), then
 * w4a16_topk of y. Every argument is checked before the first launch.
 */
int w4a16_gemm_topk(const uint16_t *x, const void *packed, int M, int N, int K, int group, int sym, int k,
                    uint16_t *y, int64_t *idx, uint16_t *vals, w4a16_stream_t stream);

/*
 * Fused feed-forward gate (GRIMOIRE v1.8, "INT4 prompt processing"):
 *   h[M][N_each] = SiLU(x Wg^T) * (x Wu^T),  SiLU(v) = v / (1 + e^-v),
 * with both products accumulated in float32 and never rounded before the
 * SiLU and the product; h is rounded once to bf16. `packed_gateup` comes from
 * w4a16_repack_gateup. Any M >= 1.
 */
int w4a16_gateup_silu(const uint16_t *x, const void *packed_gateup, int M, int N_each, int K,
                      int group, int sym, uint16_t *h, w4a16_stream_t stream);

/*
 * Test export: w_out[N][K] (float32, row-major) = (q - z) * scale read back
 * from a repacked buffer through the kernels' own unpack (exact), or, for
 * sym = W4A16_AFFINE, scale * q + bias rounded once to float32.
 */
int w4a16_dequantize(const void *packed, int N, int K, int group, int sym, float *w_out,
                     w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * Affine form: w[n][k] = scale[n][k/G] * q[n][k] + bias[n][k/G]
 * (TensorFold PR #859, "What this changes" and the AffineN notes). Every
 * code is used exactly; the products x * q are summed per group on the
 * tensor cores in float32 and each group adds scale * sum + bias * X[g][m],
 * X[g][m] = sum over the group of x[m][k]. Sizes, alignment, streams and
 * errors as for the calls above.
 * ------------------------------------------------------------------------ */

/*
 * Offline repack of an affine weight: qweight as above, scales and biases
 * bf16 [N][K/G]. The biases sit in the scales' tiled layout, and once more as
 * the tcgen05 GEMM's bias operand: bf16 [rows][kb3] with each bias at three
 * consecutive columns (against the three parts of the x group sums). Writes
 * w4a16_repacked_bytes(N, K, group, W4A16_AFFINE) bytes; padding rows get
 * code 0, scale 0 and bias 0.
 */
int w4a16_repack_affine(const int32_t *qweight, const uint16_t *scales, const uint16_t *biases, int N, int K,
                        int group, void *packed, w4a16_stream_t stream);

/* The gate/up pair of w4a16_repack_gateup in the affine form. */
int w4a16_repack_affine_gateup(const int32_t *qw_gate, const uint16_t *sc_gate, const uint16_t *b_gate,
                               const int32_t *qw_up, const uint16_t *sc_up, const uint16_t *b_up, int N_each,
                               int K, int group, void *packed, w4a16_stream_t stream);

/*
 * Group sums of the activations, X[m][g] = sum_{k in group g} x[m][k] summed
 * in float32, each stored as three bf16 parts that add up to it exactly
 * (hi = bf16(X), mid = bf16(X - hi), lo = X - hi - mid): bf16 [M][kb3],
 * kb3 = 3 * K/G rounded up to 64, the parts of X[m][g] at columns 3g .. 3g+2,
 * zeros beyond 3 * K/G. The tcgen05 GEMM multiplies them by the weight's
 * biases on the tensor cores (exact bf16 products, float32 sums). They depend
 * on x alone, so one table serves every affine weight that reads the same x
 * with the same group size. `xsum` is caller-owned device memory of
 * w4a16_xsum_bytes(M, K, group) bytes, 16-byte aligned; w4a16_xsum_bytes
 * returns 0 for unsupported sizes.
 */
size_t w4a16_xsum_bytes(int M, int K, int group);
int w4a16_xsum(const uint16_t *x, int M, int K, int group, uint16_t *xsum, w4a16_stream_t stream);

/*
 * y[M][N] (bf16) = x . (scale * q + bias)^T, W from w4a16_repack_affine.
 * `xsum` (w4a16_xsum of the same x, K and group, complete when the stream
 * reaches this call) is read by the tcgen05 GEMM (M > 32); it may be NULL
 * when M <= 32, where the decode kernel forms the group sums itself with one
 * more tensor-core product per 16 k (then it is not read).
 */
int w4a16_gemm_affine(const uint16_t *x, const uint16_t *xsum, const void *packed, int M, int N, int K, int group,
                      uint16_t *y, w4a16_stream_t stream);

/*
 * w4a16_gemm_affine without the caller's group-sum table: this library's own
 * addition, with no counterpart on the pages the method comes from. For
 * M > 32 the group sums go to a fixed 4 MiB device array inside the library's
 * module image (one per device, found once with cudaGetSymbolAddress), so the
 * call allocates nothing and needs no workspace argument; sizes whose table
 * (w4a16_xsum_bytes) exceeds 4 MiB are W4A16_ERR_INVALID_ARG (at K = 5120 and
 * group 64, M up to 8,192). Every entry the GEMM reads, the zero padding
 * included, is written by the call itself before the GEMM reads it, so
 * nothing has to start at zero. The array is shared: calls in flight at the
 * same time on one device (other streams, other host threads) race on it and
 * may compute wrong results; calls in order on one stream are safe. M <= 32
 * uses no table and behaves exactly as w4a16_gemm_affine.
 */
int w4a16_gemm_affine_noalloc(const uint16_t *x, const void *packed, int M, int N, int K, int group, uint16_t *y,
                              w4a16_stream_t stream);

/* h = SiLU(x Wg^T) * (x Wu^T) as w4a16_gateup_silu, affine weights from
 * w4a16_repack_affine_gateup; `xsum` as for w4a16_gemm_affine. */
int w4a16_gateup_silu_affine(const uint16_t *x, const uint16_t *xsum, const void *packed_gateup, int M, int N_each,
                             int K, int group, uint16_t *h, w4a16_stream_t stream);

/* ------------------------------------------------------------------------
 * Affine form at other code widths: modules of 2 to 8 bits, every code
 * keeping its value, scale and bias (TensorFold PR #859, "What this changes"
 * and the native 2, 3, 5 and 6-bit tiles note): w = scale * q + bias with q in
 * 0 .. 2^bits - 1.
 *
 * Canonical qweight: uint32 [N][ceil(K * bits / 32)], one little-endian bit
 * stream per row, code k at bits [bits * k, bits * k + bits) of the row's
 * stream (running into the next word where it does not fit); at 4 bits this
 * is the nibble packing above. scales, biases: bf16 [N][K/G].
 *
 * The repacked weight reuses the 4-bit affine kernels exactly: 2- and 3-bit
 * codes are widened into the 4-bit tiles (4 bits of memory per code); 5- to
 * 8-bit codes q = 16 qh + ql become two nibble planes over K' = 2K, group g's
 * high plane (codes qh, scale 16 * scale, the bias) followed by its low plane
 * (codes ql, the scale, bias 0), multiplied by x's group g twice (8 bits of
 * memory per code). 16 * scale is exact in bf16 for |scale| < 2^123.
 * ------------------------------------------------------------------------ */

/* Bytes of the repacked b-bit weight (0 for bits outside 2..8 or unsupported sizes). */
size_t w4a16_affine_bits_repacked_bytes(int N, int K, int group, int bits);

/* Offline repack of a b-bit affine weight; packed 256-byte aligned. */
int w4a16_repack_affine_bits(const uint32_t *qweight, const uint16_t *scales, const uint16_t *biases, int N, int K,
                             int group, int bits, void *packed, w4a16_stream_t stream);

/*
 * Bytes of the caller-owned scratch a w4a16_gemm_affine_bits call needs
 * (never 0 for supported sizes; 0 means unsupported): for 5-8 bits x with
 * each group written twice, bf16 [M][2K] (256-byte aligned), then the table of
 * x group sums of w4a16_xsum for the widened K (written when M > 32).
 */
size_t w4a16_affine_bits_scratch_bytes(int M, int K, int group, int bits);

/*
 * y[M][N] (bf16) = x . (scale * q + bias)^T for a weight from
 * w4a16_repack_affine_bits. `scratch`: w4a16_affine_bits_scratch_bytes(M, K,
 * group, bits) bytes of device memory, 256-byte aligned, used only by this
 * call while it runs on `stream` (calls in flight at once need their own).
 * Launches: the widened x (5-8 bits), the group sums (M > 32), the affine
 * GEMM. The output meets the same bound as the 4-bit form.
 */
int w4a16_gemm_affine_bits(const uint16_t *x, void *scratch, const void *packed, int M, int N, int K, int group,
                           int bits, uint16_t *y, w4a16_stream_t stream);

/* Test export: w_out[N][K] (float32) = scale * q + bias of the repacked b-bit
 * weight, rounded once to float32, q read back from its nibble planes. */
int w4a16_dequantize_affine_bits(const void *packed, int N, int K, int group, int bits, float *w_out,
                                 w4a16_stream_t stream);

/*
 * Waits for all work on the current device, then reads and clears the
 * device error word that a kernel sets when one of its bounded waits gave up
 * (W4A16_ERR_TIMEOUT; the kernel's outputs are then undefined). W4A16_OK
 * when no kernel gave up since the last call.
 */
int w4a16_kernel_status(void);

/* Static string for a status code. */
const char *w4a16_strerror(int status);

/* cudaError_t of the last W4A16_ERR_CUDA on this thread (0 if none). */
int w4a16_last_cuda_error(void);

/*
 * Kernel selection override for A/B measurement: 0 = automatic (default),
 * 1 = force the CUDA-core one-row GEMV for M = 1 (zero-point forms), 2 = force
 * the small-M tensor-core kernel with per-warp weight rings for M <= 32, 3 =
 * force the tcgen05 GEMM for any M, 4 = force the small-M kernel that stages x
 * once per CTA for M <= 16 (automatic choice: M <= 8 calls whose grid of
 * 128-row CTAs fills the GPU, e.g. the output-vocabulary head), 5 = force the
 * tcgen05 decode kernel (weights dequantised into tensor memory) for plain
 * zero-point and symmetric w4a16_gemm calls with M <= 32.
 * Returns the previous value. Process-wide; not thread-safe against
 * concurrent calls.
 */
int w4a16_set_kernel_override(int which);

/*
 * Programmatic overlap of consecutive decode calls (M <= 32), off by default.
 * When on, the M <= 32 kernels are launched with programmatic stream
 * serialization: a call may start while the previous kernel on its stream is
 * still running, begin streaming its packed weights (and scales and zeros)
 * at once, and wait for that kernel to finish (and its writes to become
 * visible) before it reads x or writes y / h. This hides each call's launch
 * and weight-fetch ramp behind the tail of the call before it, the common
 * case of decode layers run back to back (also inside CUDA graphs).
 * Turn it on only while the packed buffers are read-only: written once (at
 * load time, e.g. by w4a16_repack), then made complete by a synchronization
 * (cudaStreamSynchronize or an event the stream waits on) before the first
 * call that uses them, because the weight reads of a call are not ordered
 * after kernels still in flight on its stream. Process-wide; the setting is
 * read when a call is launched. Returns the previous setting (0 or 1), or -1
 * for a value other than 0 or 1.
 */
int w4a16_set_programmatic_overlap(int on);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H_ */
