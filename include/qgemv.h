/*
 * qgemv.h - C ABI of libqgemv.so: the weight-streaming matrix-vector product of
 * an LLM decode step over Q8_0 block-quantized weights, its bf16 variant, the
 * activation quantizers that feed it, and the prompt-sized (M rows) form of the
 * same contraction.  GB300 (sm_103a) only.
 *
 * Sources (web pages; sections as named on the page):
 *   [Phobos]  "Filling in the blanks: Inference using Phobos"
 *   [Herbert] "One level down: #002 the same compiler on a GPU"
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *   never allocates, frees or synchronises inside these calls and reads no
 *   environment variable, so every call can be recorded into a CUDA graph.
 * - Sizes are element counts.  K (the reduction length) must be a positive
 *   multiple of 32 for Q8_0 data.  A size of 0 rows is valid and launches nothing.
 * - Q8_0 weights are held as two planes ("packed layout"): values
 *   qs[n_rows][k] (int8, row-major) and scales d[n_rows][k/32] (IEEE binary16
 *   bit patterns, row-major).  qg_q8_0_pack converts the canonical 34-byte
 *   block layout into these planes.
 * - Q8_0 activations use the same two planes: q[rows][k] and d[rows][k/32].
 * - Alignment: weight value planes (qs) must be 32-byte aligned; every other
 *   pointer 16-byte aligned, except binary16 scale planes (2-byte aligned).
 * - Calls are asynchronous in the order of `stream` (NULL = legacy default
 *   stream).  Kernels are launched with programmatic dependent launch: a kernel
 *   may start streaming its WEIGHTS while the previous kernel in the stream
 *   finishes, and reads activations only after that kernel has completed.
 *   Weights must therefore not be written by a kernel that is still running
 *   when the call is made (writes by qg_q8_0_pack or by any kernel that has
 *   completed are fine).
 * - Errors: argument errors are returned before anything is launched; a
 *   launch failure returns QG_ERR_CUDA.  Errors inside the kernels are not
 *   reported by these calls (the kernels have no failing paths on valid input),
 *   except by qg_decode_stack_q8_0, whose workspace holds a status word.
 * - Outputs never alias inputs, except where a call says so.
 * - Threads and state: calls may be made from several host threads.  The
 *   library keeps per-device caches, filled on first use under a lock (the SM
 *   count, the shared-memory opt-in of each kernel).  Two entry points share
 *   device memory between calls: qg_decode_layers_q8_0_noalloc uses one fixed
 *   array per GPU compiled into the library, and qg_decode_stack_q8_0 a
 *   caller-owned workspace.  Calls that share that array, or a workspace, must
 *   not overlap in time; every other call is independent of every other.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stdint.h>

#if defined(__GNUC__)
#define QG_API __attribute__((visibility("default")))
#else
#define QG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *qg_stream_t;

typedef enum {
    QG_OK = 0,
    QG_ERR_NULL = 1,        /* a required pointer is NULL */
    QG_ERR_ALIGN = 2,       /* a pointer breaks the alignment rule above */
    QG_ERR_SHAPE = 3,       /* a size is negative, not a multiple of 32, or too large */
    QG_ERR_UNSUPPORTED = 4, /* valid request this build does not serve (e.g. batch > 8) */
    QG_ERR_CUDA = 5         /* the CUDA runtime reported an error at launch */
} qg_status;

/* Epilogues fused into the GEMV ([Phobos] Fast Decode: fold the residual add
 * into the matmul; [Herbert] Emitting for a GPU: the activation is fused with
 * the projection). */
typedef enum {
    QG_EPI_NONE = 0,            /* y[b][n] = dot(W[n], x[b]) */
    QG_EPI_SILU_MUL_HALVES = 1, /* n_rows even, F = n_rows/2, rows [0,F) gate, [F,2F) up:
                                   y[b][i] = silu(g_i) * u_i, silu(g) = g / (1 + e^-g),
                                   y has F columns per batch row */
    QG_EPI_RESIDUAL_ADD = 2     /* y[b][n] = residual[b][n] + dot(W[n], x[b]);
                                   residual may be the same buffer as y */
} qg_epilogue;

/* Human-readable name of a status. */
QG_API const char *qg_status_str(qg_status s);

/* ABI version of this header (bumped on any signature change). */
QG_API int qg_abi_version(void);

/*
 * qg_q8_0_pack - canonical Q8_0 blocks -> packed planes.
 * [Phobos] GPU Performance Heisenbugs: weights are stored so that a decode warp
 * reads whole cache lines.  Canonical block: 2-byte little-endian binary16 scale
 * followed by 32 int8 values (34 bytes); blocks[n_rows][k/32].
 *   blocks: device, 1-byte aligned, n_rows*(k/32)*34 bytes (read)
 *   qs:     device, 32-byte aligned, int8[n_rows][k] (written)
 *   d:      device, binary16 bits uint16[n_rows][k/32] (written)
 * A byte permutation; a one-time load step, not part of the decode step.
 */
QG_API qg_status qg_q8_0_pack(const void *blocks, int64_t n_rows, int64_t k,
                       int8_t *qs, uint16_t *d, qg_stream_t stream);

/*
 * qg_q8_0_column_blocks - re-lay packed Q8_0 planes column block by column
 * block: block b of row n moves to qs_cb[b][n][0..31] and its scale to
 * d_cb[b][n], so all rows of one 32-column block are contiguous.  The pages lay
 * weights out for the kernel that reads them ([Phobos] GPU Performance
 * Heisenbugs: groups of eight columns); this is the layout of the down weights
 * of qg_decode_layer_q8_0, whose CTAs each read one column block of every row.
 *   qs: device int8[n_rows][k] (read), 32-byte aligned; d: binary16 [n_rows][k/32]
 *   qs_cb: device int8[k/32][n_rows][32] (written), 32-byte aligned
 *   d_cb: device binary16 [k/32][n_rows] (written)
 *   Outputs must not overlap inputs (QG_ERR_SHAPE).  A one-time load step; like
 *   qg_q8_0_pack it does not let the next kernel start reading weights early.
 */
QG_API qg_status qg_q8_0_column_blocks(const int8_t *qs, const uint16_t *d, int64_t n_rows,
                                       int64_t k, int8_t *qs_cb, uint16_t *d_cb,
                                       qg_stream_t stream);

/*
 * quantize_act_q8_0 - quantize activations to Q8_0, once, to be shared by
 * every projection that reads them ([Phobos] Fast Decode).
 * Per 32-value block: d = max|x| / 127 (f32), q = round half away from zero of
 * x / d (one IEEE f32 division; d == 0 gives q = 0), clamped to [-127, 127];
 * the stored scale is binary16(d), round to nearest even.
 *   x: device f32[rows][k] (read)
 *   q: device int8[rows][k] (written)      d: device binary16 bits [rows][k/32] (written)
 */
QG_API qg_status quantize_act_q8_0(const float *x, int64_t rows, int64_t k,
                            int8_t *q, uint16_t *d, qg_stream_t stream);

/*
 * quantize_act_q8_0_tiles - the Q8_0 quantization of quantize_act_q8_0 (same
 * codes, same scales), written as the activation operand of the tensor-core
 * prompt contraction qgemm_q8_0_prefill_tc ([Phobos] Fast Decode: prompt
 * processing runs on the tensor cores).  The pages store codes as int8; this
 * form holds each code as a binary16 value (exact: an integer in [-127, 127])
 * already in the order the tensor core reads, so the contraction copies it
 * without conversion.
 *   Layout: rows in tiles of 128 (rows past `rows` in the last tile are zero);
 *   for tile t and block j one record of 8448 bytes at byte offset
 *   (t * (k/32) + j) * 8448:
 *     bytes [0, 8192):    code 8g+e (g < 4, e < 8) of tile row r as binary16 at
 *                         byte 2048 g + 16 r + 2 e;
 *     bytes [8192, 8448): the 128 binary16 scales of the tile rows.
 *   x:  device f32[rows][k] (read), 16-byte aligned; rows <= 2^24
 *   xt: device, qg_act_tiles_bytes(rows, k) bytes (written), 16-byte aligned;
 *       caller-owned.
 */
QG_API int64_t qg_act_tiles_bytes(int64_t rows, int64_t k);  /* -1: shape unsupported */
QG_API qg_status quantize_act_q8_0_tiles(const float *x, int64_t rows, int64_t k, void *xt,
                                         qg_stream_t stream);

/*
 * rmsnorm_quantize - RMSNorm followed by Q8_0 quantization of each row.
 * [Herbert] Emitting for a GPU (normalization fused with the projection that
 * follows it); [Phobos] Q4_K_M (the fast norm kernel).
 *   r = 1 / sqrt(mean_k(x^2) + eps), evaluated in f64 and rounded once to f32;
 *   x_hat = (x * r) * gamma (two f32 multiplies); then quantize_act_q8_0(x_hat).
 *   x:       device f32[rows][k] (read)     gamma: device f32[k] (read)
 *   q, d:    as quantize_act_q8_0 (written)
 *   inv_rms: device f32[rows] receiving r, or NULL
 *   k <= 65536.
 */
QG_API qg_status rmsnorm_quantize(const float *x, const float *gamma, int64_t rows, int64_t k,
                           float eps, int8_t *q, uint16_t *d, float *inv_rms,
                           qg_stream_t stream);

/*
 * rmsnorm_hadamard_quantize - rmsnorm_quantize with the normalised row rotated
 * before it is quantized ([Phobos] PrismML Ternary-Bonsai-2-27B: a Hadamard
 * matrix transform rotates the activation over the format's block, spreading
 * outliers over it; the rotated activation is computed once and shared by every
 * projection that reads the same input, whose weights carry the inverse
 * rotation from load time: W x_hat = (W H^T / 128)(H x_hat)).  Per row:
 *   r, x_hat = (x * r) * gamma            exactly as rmsnorm_quantize
 *   z[128 b + i] = sum_j (-1)^popcount(i & j) x_hat[128 b + j]
 *       (Walsh-Hadamard matrix of order 128, Sylvester order, unnormalised,
 *        on each block of 128; summed in f32 by the fast transform's
 *        butterflies, strides 1, 2, 4, ..., 64 in that order)
 *   q, d   = Q8_0(z)                        (as quantize_act_q8_0 of z)
 *   x, gamma: f32[rows][k] / f32[k], 16-byte aligned; k a multiple of 128 up to
 *   65536; q: int8[rows][k] (16-byte aligned); d: binary16[rows][k/32];
 *   z: optional f32[rows][k] (16-byte aligned) receiving the rotated row;
 *   inv_rms: optional f32[rows].  Errors as rmsnorm_quantize.
 */
QG_API qg_status rmsnorm_hadamard_quantize(const float *x, const float *gamma, int64_t rows, int64_t k,
                                           float eps, int8_t *q_out, uint16_t *d_out, float *z_out,
                                           float *inv_rms_out, qg_stream_t stream);

/*
 * qgemv_q8_0 - block-scaled Q8_0 matrix-vector product ([Phobos] Fast Decode:
 * int8 dot products end to end, one scale per 32 values, a warp owns an output
 * row and reduces with shuffles).
 *   acc[b][n] = sum over blocks j of f32(d_w[n][j]) * f32(d_x[b][j]) * S_j,
 *   S_j = exact int32 sum of w_qs[n][32j+i] * xq[b][32j+i], i < 32;
 *   accumulation in f32 (order unspecified), then the epilogue.
 *   w_qs, w_d: packed weight planes [n_rows][k], [n_rows][k/32] (read)
 *   xq, xd:    Q8_0 activations [batch][k], [batch][k/32] (read)
 *   batch:     1 <= batch <= 8 (batch rows share one pass over the weights)
 *   epilogue:  a qg_epilogue; residual: device f32[batch][n_rows] for
 *              QG_EPI_RESIDUAL_ADD (may equal y), else ignored
 *   y:         device f32[batch][n_out], n_out = n_rows, or n_rows/2 for
 *              QG_EPI_SILU_MUL_HALVES (written)
 */
QG_API qg_status qgemv_q8_0(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows, int64_t k,
                     const int8_t *xq, const uint16_t *xd, int64_t batch,
                     int epilogue, const float *residual, float *y, qg_stream_t stream);

/*
 * qgemv_bf16 - bf16-weight matrix-vector product with f32 accumulation
 * ([Herbert] The numerical contract; Emitting for a GPU: rows read as 16-byte
 * groups of eight bf16, norm fused in front, activation fused behind).
 *   With gamma != NULL: r = 1/sqrt(mean(x^2)+eps) (f64, rounded to f32),
 *   x_hat = bf16_rne((x * r) * gamma); with gamma == NULL: x_hat = x.
 *   acc[n] = sum_k f32(w[n][k]) * f32(x_hat[k]) in f32, then the epilogue
 *   (QG_EPI_NONE, QG_EPI_SILU_MUL_HALVES or QG_EPI_RESIDUAL_ADD as above).
 *   w: device bf16 bits [n_rows][k] (read), k a multiple of 8, k <= 16384
 *   x, gamma: device bf16 bits [k] (read)
 *   y: device f32[n_out] (written)
 *   Each output is summed in one fixed order whatever the shape.
 */
QG_API qg_status qgemv_bf16(const uint16_t *w, int64_t n_rows, int64_t k, const uint16_t *x,
                     const uint16_t *gamma, float eps, int epilogue,
                     const float *residual, float *y, qg_stream_t stream);

/*
 * qgemm_q8_0_prefill - the same block-scaled contraction for M prompt rows
 * ([Phobos] Fast Decode: prompt processing reuses every weight M times and
 * belongs on the tensor cores; GPU Performance Heisenbugs: exact int8 values
 * run straight on the integer tensor cores).
 *   Y[m][n] = sum_j f32(d_x[m][j]) * f32(d_w[n][j]) * S_j[m][n], f32 accumulation.
 *   xq, xd: Q8_0 activations [m][k], [m][k/32]; w_qs, w_d: packed weights.
 *   y: device f32[m][n_rows] (written)
 */
QG_API qg_status qgemm_q8_0_prefill(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows,
                             int64_t k, const int8_t *xq, const uint16_t *xd, int64_t m,
                             float *y, qg_stream_t stream);

/*
 * qg_ffn_up_q8_0 - the first half of a decode feed-forward block in one launch:
 * RMSNorm of x, Q8_0 quantization of x_hat, the stacked gate|up product, and
 * SiLU(g) * u, whose 32-value blocks are quantized to Q8_0 on the way out.
 * [Phobos] Fast Decode (quantize once and share; stack projections that read
 * the same input); [Herbert] Emitting for a GPU (normalization fused with the
 * projection that follows it, activation fused with the projection before it).
 *   Arithmetic identical to rmsnorm_quantize -> qgemv_q8_0(SILU_MUL_HALVES)
 *   -> quantize_act_q8_0, bit for bit.
 *   x: device f32[hidden] (read); gamma: device f32[hidden] (read)
 *   w_qs, w_d: stacked gate|up weight planes [2*ffn][hidden], [2*ffn][hidden/32]
 *   h: device f32[ffn] (written); hq: int8[ffn], hd: binary16 bits [ffn/32] (written)
 *   xq_out, xd_out, inv_rms_out: optional copies of the quantized input and of r
 *   hidden % 256 == 0 and hidden <= 2048; ffn % 32 == 0 (else QG_ERR_UNSUPPORTED
 *   or QG_ERR_SHAPE); w_d 16-byte aligned.
 */
QG_API qg_status qg_ffn_up_q8_0(const float *x, const float *gamma, int64_t hidden, float eps,
                                const int8_t *w_qs, const uint16_t *w_d, int64_t ffn,
                                float *h, int8_t *hq, uint16_t *hd, int8_t *xq_out,
                                uint16_t *xd_out, float *inv_rms_out, qg_stream_t stream);

/*
 * qg_decode_ffn_q8_0 - one decode feed-forward block, x <- x + down(h), in two
 * launches: qg_ffn_up_q8_0, then qgemv_q8_0(down, hq, hd, QG_EPI_RESIDUAL_ADD)
 * in place on x ([Phobos] Fast Decode: fold the residual add into the matmul).
 *   x: device f32[hidden], read and overwritten with the block's output
 *   wgu_*: stacked gate|up planes [2*ffn][hidden]; wdn_*: down planes [hidden][ffn]
 *   h, hq, hd: caller-owned work buffers f32[ffn], int8[ffn], binary16[ffn/32]
 *              (left holding this block's activation); hq 32-byte aligned
 *   shapes as qg_ffn_up_q8_0; both scale planes 16-byte aligned.
 */
QG_API qg_status qg_decode_ffn_q8_0(float *x, const float *gamma, int64_t hidden, int64_t ffn,
                                    float eps, const int8_t *wgu_qs, const uint16_t *wgu_d,
                                    const int8_t *wdn_qs, const uint16_t *wdn_d, float *h,
                                    int8_t *hq, uint16_t *hd, qg_stream_t stream);

/*
 * qg_decode_ffn_q8_0_out - the same block out of place: x_out = x_in + down(h),
 * h computed from x_in.  x_in and x_out are the same pointer (in place, as
 * qg_decode_ffn_q8_0) or do not overlap (QG_ERR_SHAPE otherwise); both are f32
 * [hidden], 16-byte aligned, and may be device memory or pinned host memory
 * (read or written by the kernels directly over the host link), so a step can
 * take its input from, and leave its result in, host buffers without separate
 * copies.  Other arguments and errors as qg_decode_ffn_q8_0.
 */
QG_API qg_status qg_decode_ffn_q8_0_out(const float *x_in, float *x_out, const float *gamma, int64_t hidden,
                                        int64_t ffn, float eps, const int8_t *wgu_qs, const uint16_t *wgu_d,
                                        const int8_t *wdn_qs, const uint16_t *wdn_d, float *h, int8_t *hq,
                                        uint16_t *hd, qg_stream_t stream);

/*
 * qg_decode_ffn_q8_0_rotated - qg_decode_ffn_q8_0_out with the normalised
 * activation rotated before it is quantized ([Phobos] PrismML
 * Ternary-Bonsai-2-27B: the rotated activation is computed once and shared by
 * every projection that reads the input; here by both halves of the stacked
 * gate|up), in two launches:
 *   z = H x_hat per block of 128 (as rmsnorm_hadamard_quantize: x_hat =
 *       (x r) gamma, the order-128 Walsh-Hadamard matrix, unnormalised),
 *   (g|u) = gate|up(Q8_0(z)), h = SiLU(g) u, x_out = x_in + down(Q8_0(h)).
 * The stacked gate|up weights are the rotated ones (W H^T / 128, quantized at
 * load time), so that W x_hat = (W H^T / 128) z.
 *   xq_out, xd_out: optional (NULL): the rotated activation's codes int8[hidden]
 *          (16-byte aligned) and scales binary16[hidden/32].
 *   hidden a multiple of 256 up to 1024 (one rotation block per warp); ffn as
 *   qg_decode_ffn_q8_0 with the down weights served by the staged GEMV (ffn a
 *   multiple of 256 up to 4096); other arguments and errors as
 *   qg_decode_ffn_q8_0_out.
 */
QG_API qg_status qg_decode_ffn_q8_0_rotated(const float *x_in, float *x_out, const float *gamma,
                                            int64_t hidden, int64_t ffn, float eps,
                                            const int8_t *wgu_qs, const uint16_t *wgu_d,
                                            const int8_t *wdn_qs, const uint16_t *wdn_d, float *h,
                                            int8_t *hq, uint16_t *hd, int8_t *xq_out, uint16_t *xd_out,
                                            qg_stream_t stream);

/*
 * qg_decode_layer_q8_0 - one decode feed-forward block in ONE launch, its
 * input and output each held unreduced as a base vector plus partial vectors:
 *   x      = r_in + p_in[0] + ... + p_in[n_in - 1]        (f32, in that order)
 *   r_out  = x
 *   r_out + p_out[0] + ... + p_out[P - 1] = x + down(Q8_0(SiLU(g) * u)),
 *   (g|u)  = gate|up(Q8_0(RMSNorm(x) * gamma)),  P = qg_decode_layer_partials.
 * [Phobos] Fast Decode: quantize once and share, stack the projections, fold
 * the residual into the matmul; [Herbert] Emitting for a GPU: fuse the
 * normalization and the activation with the projections around them.  The
 * pages launch the down projection separately; here it is split along its
 * reduction: the CTA that produces block b of h forms that block's Q8_0 term
 * of every output (f32(d_w[n][b]) * f32(d_h[b]) * exact block sum), the CTAs
 * of a thread-block cluster (up to 8) add their terms on chip, and each
 * cluster stores one partial output vector.  The next layer sums them while
 * it loads its input, so no pass over the output and no atomics are needed;
 * every sum is in a fixed order, so results repeat bit for bit.
 *   r_in:  device f32[hidden] (read), 16-byte aligned
 *   p_in:  device f32[n_in][hidden] (read), 16-byte aligned; NULL when n_in = 0;
 *          n_in <= 16
 *   r_out: device f32[hidden] (written), 16-byte aligned
 *   p_out: device f32[P][hidden] (written), 16-byte aligned
 *          No output may overlap an input or the other output (QG_ERR_SHAPE).
 *   gamma, wgu_*, h, hq, hd: as qg_decode_ffn_q8_0 (h, hq, hd left holding
 *          this block's activation).
 *   wdn_qs, wdn_d: the down weights in the column-block layout written by
 *          qg_q8_0_column_blocks: values int8[ffn/32][hidden][32] (32-byte
 *          aligned), scales binary16[ffn/32][hidden] (16-byte aligned).
 *   hidden a multiple of 256 whose one-launch working set fits one CTA's shared
 *   memory (hidden <= 2048 on GB300); ffn a multiple of 32 with P <= 16
 *   (QG_ERR_UNSUPPORTED otherwise).  A CTA whose staged copies stall beyond
 *   one second stops waiting instead of hanging: the outputs are then undefined
 *   (NaN where it can still write them) and the stall is counted
 *   (qg_copy_stalls).
 * A stack of layers ping-pongs two (r, p) pairs, layer 0 with n_in = 0, and
 * ends with qg_decode_layer_finish.
 */
QG_API qg_status qg_decode_layer_q8_0(const float *r_in, const float *p_in, int32_t n_in,
                                      float *r_out, float *p_out, const float *gamma,
                                      int64_t hidden, int64_t ffn, float eps,
                                      const int8_t *wgu_qs, const uint16_t *wgu_d,
                                      const int8_t *wdn_qs, const uint16_t *wdn_d, float *h,
                                      int8_t *hq, uint16_t *hd, qg_stream_t stream);

/* Partial vectors P a qg_decode_layer_q8_0 call writes (-1: shape unsupported). */
QG_API int32_t qg_decode_layer_partials(int64_t hidden, int64_t ffn);

/*
 * qg_decode_layer_finish - x = r + p[0] + ... + p[n - 1] (f32, in that order,
 * the order the next layer would use): the output of a stack of one-launch
 * layers as one vector.
 *   r: device f32[hidden]; p: device f32[n][hidden] (NULL when n = 0), n <= 16;
 *   x: device f32[hidden] (written; may be r itself).
 */
QG_API qg_status qg_decode_layer_finish(const float *r, const float *p, int32_t n, int64_t hidden,
                                        float *x, qg_stream_t stream);

/*
 * qg_copy_stalls - how many waits of the decode kernels on their staged weight
 * copies gave up (after one second) on the current device since the last clear:
 * a CTA of the gate|up kernel (qg_ffn_up_q8_0, the qg_decode_ffn_q8_0 family,
 * qg_decode_layer_q8_0, the layers of qg_decode_layers_q8_0_noalloc) or a warp of
 * the staging GEMV (their down projection, and qgemv_q8_0 at batch 1 where the
 * weights fit one wave) counts one.  The outputs of a call with such a stall are
 * undefined (NaN where the kernel could still write them); 0 in normal
 * operation.  Not a hang detector for the persistent stack, which reports
 * through its workspace status word.
 *   count: host uint32_t (written).  clear != 0 resets the counter after reading.
 * Reads device memory with a synchronous copy: it waits for the device's work.
 */
QG_API qg_status qg_copy_stalls(uint32_t *count, int32_t clear);

/*
 * qg_decode_layers_q8_0_noalloc - a stack of n_layers one-launch decode layers
 * (qg_decode_layer_q8_0 for each, then qg_decode_layer_finish into x_out) that
 * needs no caller-provided work memory.  The pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory.  The
 * layers' intermediates (the unreduced inputs and outputs, h and its codes)
 * live in one fixed array compiled into the library, 256 KB per GPU; shapes
 * whose intermediates do not fit it are refused with QG_ERR_UNSUPPORTED
 * (hidden 1024 / ffn 3584 needs 141,056 bytes; hidden 1792 / ffn 4096 does
 * not fit).  Results are the same bits as
 * running the layers through qg_decode_layer_q8_0 with caller buffers.
 *   x_in:  device f32[hidden] (read), 16-byte aligned
 *   x_out: device f32[hidden] (written); may be x_in
 *   gamma, wgu_qs, wgu_d, wdn_qs, wdn_d: HOST arrays of n_layers DEVICE
 *          pointers, one set per layer, as qg_decode_layer_q8_0 (down weights
 *          in the column-block layout of qg_q8_0_column_blocks); read during
 *          the call only.
 *   hidden, ffn, eps: as qg_decode_layer_q8_0, the same for every layer.
 * Concurrency: the array is shared by every call on a GPU, so calls on the same
 * GPU must not overlap in time (one stream, or synchronise between them).
 * The first call on each GPU looks the array up (a host-side query): make it
 * before capturing the call into a CUDA graph.
 */
QG_API qg_status qg_decode_layers_q8_0_noalloc(const float *x_in, float *x_out, int32_t n_layers,
                                               const float *const *gamma,
                                               const int8_t *const *wgu_qs, const uint16_t *const *wgu_d,
                                               const int8_t *const *wdn_qs, const uint16_t *const *wdn_d,
                                               int64_t hidden, int64_t ffn, float eps,
                                               qg_stream_t stream);

/*
 * qg_decode_stack_q8_0 - n_layers decode feed-forward blocks, each
 *   x <- x + down(Q8_0(SiLU(g) * u)),  (g|u) = gate|up(Q8_0(RMSNorm(x) * gamma)),
 * in ONE persistent launch ([Phobos] Q4_K_M: the whole MLP as one persistent
 * kernel; Fast Decode: quantize the activation once and share it, stack the
 * projections, fold the residual into the matmul; [Herbert] Emitting for a GPU:
 * fuse the normalization and the activation with the projections around them).
 * One CTA per SM, launched cooperatively (all resident at once); each layer's
 * two all-to-all steps (all of x before the gate|up rows, all of h before the
 * down rows) are hand-offs through workspace words that hold a value and an
 * epoch, polled by the consumers, instead of kernel boundaries; the weights of
 * the next layers stream into shared memory while a layer computes.  The
 * result has the same bits as n_layers calls of qg_decode_ffn_q8_0_out.
 *   x_in:  f32[hidden], 16-byte aligned: device or pinned host memory (read)
 *   x_out: f32[hidden]: device or pinned host memory (written); x_in itself,
 *          or not overlapping it (QG_ERR_SHAPE otherwise)
 *   gamma, wgu_qs, wgu_d, wdn_qs, wdn_d: HOST arrays of n_layers DEVICE
 *          pointers, one set per layer, read during the call only: gains
 *          f32[hidden] (16-byte aligned), stacked gate|up planes [2*ffn][hidden],
 *          down planes [hidden][ffn] (row-major, as qg_decode_ffn_q8_0; values
 *          32-byte, scales 16-byte aligned)
 *   n_layers: 1 .. qg_decode_stack_max_layers() (QG_ERR_SHAPE otherwise);
 *          chain calls for more layers (x_out of one as x_in of the next)
 *   workspace: device memory of qg_decode_stack_workspace_bytes(hidden, ffn)
 *          bytes, 256-byte aligned, ZERO-FILLED before its first use and then
 *          left to the library; one workspace serves one shape; calls that
 *          share a workspace must not overlap in time (one stream).  Its first
 *          32-bit word is the status: 0 while every launch since it was zeroed
 *          completed normally; bit 0 set when a hand-off wait ran past
 *          wait_limit_ns (or saw another CTA give up), bit 1 when a weight copy
 *          did not land in time.  A launch that sets it returns normally with
 *          x_out (and h_last) undefined; the status stays set until the
 *          workspace is zero-filled again.
 *   h_last, hq_last, hd_last: optional (NULL): the last layer's h f32[ffn]
 *          (4-byte aligned), its Q8_0 codes int8[ffn] and scales binary16[ffn/32]
 *   wait_limit_ns: bound on every wait inside the kernel; 0 = one second
 *   Shapes: hidden a multiple of 256 up to 1024, ffn a multiple of 256 up to
 *   4096 with ffn/32 at most the SM count, and both layers' weight slabs within
 *   one CTA's shared memory (QG_ERR_UNSUPPORTED otherwise; the 0.8B shape,
 *   hidden 1024 / ffn 3584, is served).  A failed cooperative launch (e.g. SMs
 *   held by other work) returns QG_ERR_CUDA.
 */
QG_API int64_t qg_decode_stack_workspace_bytes(int64_t hidden, int64_t ffn); /* -1: unsupported */
QG_API int32_t qg_decode_stack_max_layers(void);
QG_API qg_status qg_decode_stack_q8_0(const float *x_in, float *x_out, int32_t n_layers,
                                      const float *const *gamma,
                                      const int8_t *const *wgu_qs, const uint16_t *const *wgu_d,
                                      const int8_t *const *wdn_qs, const uint16_t *const *wdn_d,
                                      int64_t hidden, int64_t ffn, float eps, void *workspace,
                                      float *h_last, int8_t *hq_last, uint16_t *hd_last,
                                      int64_t wait_limit_ns, qg_stream_t stream);

/*
 * qgemm_q8_0_prefill_tc - the prompt contraction of qgemm_q8_0_prefill on the
 * tcgen05 tensor cores ([Phobos] Fast Decode: prompt processing belongs on the
 * tensor cores; GPU Performance Heisenbugs: exact integer values on the tensor
 * cores).  Exact int8 codes run as f16 operands, the exact block sums land in
 * the f32 accumulator, and the block scales are applied per block:
 *   Y[m][n] = sum_j f32(d_x[m][j]) * f32(d_w[n][j]) * S_j[m][n].
 *   w_qs: device int8[n_rows][k] (read), 32-byte aligned
 *   w_d:  device binary16 bits [n_rows][k/32] (read), 16-byte aligned
 *   xt:   activation tiles of m rows from quantize_act_q8_0_tiles (read)
 *   y:    device f32[m][n_rows] (written), 16-byte aligned
 *   k a multiple of 256 (QG_ERR_UNSUPPORTED otherwise); m <= 2^24.
 *   tile_n: output tile width 64, 96 or 128, or 0 to let the library choose.
 *   Runs one CTA per SM over all output tiles.  If an operand copy stalls
 *   beyond one second the kernel stops waiting and writes NaN for the tiles
 *   it has left, rather than hanging.
 */
QG_API qg_status qgemm_q8_0_prefill_tc(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows,
                                       int64_t k, const void *xt, int64_t m, float *y,
                                       int32_t tile_n, qg_stream_t stream);

/*
 * qg_debug_block_dots_q8_0 - the exact per-block int32 sums, for parity checks.
 *   s[b][n][j] = sum_{i<32} w_qs[n][32j+i] * xq[b][32j+i]   (int32, exact)
 *   s: device int32[batch][n_rows][k/32] (written); batch <= 8.
 */
QG_API qg_status qg_debug_block_dots_q8_0(const int8_t *w_qs, int64_t n_rows, int64_t k,
                                   const int8_t *xq, int64_t batch, int32_t *s,
                                   qg_stream_t stream);

/*
 * Operands for qgemm_q8_0_prefill_tc2, the prompt contraction over wide tiles
 * ([Phobos] Fast Decode: prompt processing on the tensor cores; GPU Performance
 * Heisenbugs: exact integer values on the tensor cores).  Codes are held as
 * binary16 values (exact: integers in [-127, 127]) in plain row-major matrices,
 * scales as f32 block-major [k/32][ld] with ld = qg_scales_ld(rows), rows rounded
 * up to a multiple of four so that each block's row starts on 16 bytes (the
 * padding entries are neither written nor read).
 *
 * qg_q8_0_pack_f16 - weight planes -> that form (a one-time load step).
 *   w_qs: device int8 [n_rows][k] (read), 8-byte aligned; w_d: binary16 bits
 *   [n_rows][k/32] (read); codes: device binary16 [n_rows][k] (written),
 *   16-byte aligned; scales_t: device f32 [k/32][ld] (written).  k a
 *   multiple of 32.  Outputs must not overlap inputs (QG_ERR_SHAPE).
 *
 * quantize_act_q8_0_f16 - quantize_act_q8_0 (same codes, same binary16-rounded
 *   scales) writing that form: x f32 [rows][k] (read, 16-byte aligned),
 *   codes binary16 [rows][k], scales_t f32 [k/32][ld] (written).
 *
 * qgemm_q8_0_prefill_tc2 - Y[m][n] = sum_j f32(d_x[m][j]) f32(d_w[n][j]) S_j[m][n]
 *   on tcgen05 over 128 x tile_n output tiles (tile_n 128 or 192, or 0 to let
 *   the library choose): exact block sums S_j in TMEM, the rescale in f32
 *   registers.  w_codes, w_scales_t: from qg_q8_0_pack_f16; x_codes, x_scales_t:
 *   from quantize_act_q8_0_f16 for m rows; y: device f32 [m][n_rows] (written).
 *   Operands 16-byte aligned, k a multiple of 32, m <= 2^24; y must not overlap
 *   the operands (QG_ERR_SHAPE).  Runs one CTA per SM; if an operand copy stalls
 *   beyond one second the kernel writes NaN for the tiles it has left.
 */
QG_API int64_t qg_scales_ld(int64_t rows);
QG_API qg_status qg_q8_0_pack_f16(const int8_t *w_qs, const uint16_t *w_d, int64_t n_rows, int64_t k,
                                  uint16_t *codes, float *scales_t, qg_stream_t stream);
QG_API qg_status quantize_act_q8_0_f16(const float *x, int64_t rows, int64_t k, uint16_t *codes,
                                       float *scales_t, qg_stream_t stream);
QG_API qg_status qgemm_q8_0_prefill_tc2(const uint16_t *w_codes, const float *w_scales_t, int64_t n_rows,
                                        int64_t k, const uint16_t *x_codes, const float *x_scales_t,
                                        int64_t m, float *y, int32_t tile_n, qg_stream_t stream);

/*
 * qg_measure_mma_s8 - times nothing itself: launches a grid (4 CTAs per SM) whose
 * warps issue `iters` rounds of eight independent mma.sync.m16n8k32 s8 MMAs on
 * register operands, the int8 tensor path that sm_103a offers ([Phobos] GPU
 * Performance Heisenbugs: integer tensor cores), so that a caller timing the
 * stream gets that path's rate, the second roofline of the prompt contraction.
 *   iters: 1 .. 2^24; sink: device int32 (written only in an impossible case);
 *   *ops (host): the int-ops the launch performs.  Errors: QG_ERR_SHAPE,
 *   QG_ERR_NULL, QG_ERR_CUDA.
 */
QG_API qg_status qg_measure_mma_s8(int64_t iters, int32_t *sink, int64_t *ops, qg_stream_t stream);

/*
 * qg_measure_hbm_read - reads `bytes` of device memory once, from every SM, with
 * the 32-byte streaming loads of the GEMV kernels, and folds them into one word
 * per CTA of `sink`: the pure-read bandwidth probe that a decode product is
 * judged against ([Herbert] Decode: memory decides: decode matvec against a
 * pure-read probe on the same machine).  A caller times the stream.
 *   buf: device, 32-byte aligned; bytes: a positive multiple of 32;
 *   sink: device uint32[sink_len], sink_len >= qg_measure_hbm_read_sink_len().
 *   Errors: QG_ERR_SHAPE, QG_ERR_NULL, QG_ERR_ALIGN, QG_ERR_CUDA.
 */
QG_API int32_t qg_measure_hbm_read_sink_len(void);
QG_API qg_status qg_measure_hbm_read(const void *buf, int64_t bytes, uint32_t *sink, int32_t sink_len,
                                     qg_stream_t stream);

/*
 * qg_measure_launch_chain - launches n empty kernels of grid x block threads on
 * `stream`, each waiting for its predecessor and letting its successor launch
 * (programmatic dependent launch, as every kernel of the library): timed by the
 * caller, the cost of a kernel boundary alone, the floor of a GEMV whose bytes
 * take less time than its launch.  Not part of the method.
 *   n: 0 .. 65536; grid: 1 .. 65535; block: a multiple of 32 up to 1024.
 *   Errors: QG_ERR_SHAPE, QG_ERR_CUDA.
 */
QG_API qg_status qg_measure_launch_chain(int32_t n, int32_t grid, int32_t block, qg_stream_t stream);

/*
 * qgemm_bf16_prefill - qgemv_bf16 for m prompt rows at once, on the tcgen05
 * tensor cores ([Herbert] The numerical contract: bf16 weights and activations,
 * f32 accumulators; Emitting for a GPU: norm fused in front, SiLU(g)*u behind,
 * stacked gate|up; [Phobos] Fast Decode: a prompt reuses every weight for all of
 * its rows, so it runs on the tensor cores).  Row i of the result is what
 * qgemv_bf16 computes for row i of x, up to the order of the f32 sums:
 *   with gamma != NULL, per row: r = 1/sqrt(mean(x^2)+eps) (f64, rounded to f32),
 *   x_hat = bf16_rne((x * r) * gamma); with gamma == NULL, x_hat = x;
 *   acc[i][n] = sum_k f32(w[n][k]) * f32(x_hat[i][k]) in f32 (exact products);
 *   epilogue QG_EPI_NONE (y[i][n] = acc, n_out = n_rows) or
 *   QG_EPI_SILU_MUL_HALVES (y[i][j] = silu(acc[i][j]) * acc[i][j + n_rows/2],
 *   n_out = n_rows / 2, n_rows even).
 *   w: device bf16 bits [n_rows][k] (read), 16-byte aligned; k a multiple of 8,
 *      k <= 16384
 *   x: device bf16 bits [m][k] (read), 16-byte aligned; gamma: bf16 bits [k] or NULL
 *   xhat: device bf16 [m][k] work buffer, owned by the caller, written when
 *      gamma != NULL (may be NULL otherwise), 16-byte aligned, not overlapping x
 *   y: device f32 [m][n_out] (written), 16-byte aligned; m <= 2^24
 *   Outputs (y, and xhat when gamma != NULL) must not overlap the inputs or
 *   each other (QG_ERR_SHAPE).
 *   Runs one CTA per SM over 128 x 256 accumulator tiles.  If an operand copy
 *   stalls beyond one second the kernel stops waiting and writes NaN for the
 *   tiles it has left, rather than hanging.  Errors: QG_ERR_SHAPE, QG_ERR_NULL,
 *   QG_ERR_ALIGN, QG_ERR_UNSUPPORTED (epilogue QG_EPI_RESIDUAL_ADD), QG_ERR_CUDA.
 */
QG_API qg_status qgemm_bf16_prefill(const uint16_t *w, int64_t n_rows, int64_t k, const uint16_t *x,
                                    int64_t m, const uint16_t *gamma, float eps, int epilogue,
                                    uint16_t *xhat, float *y, qg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_H */
