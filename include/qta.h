/*
 * qta.h -- C ABI of the quantized tensor-activation codec for GB300 (sm_103a).
 *
 * The library compresses tensor-parallel activations / gradients before a
 * collective and performs the dequantize -> FP32 reduce -> requantize math of
 * a quantized reduce-scatter / all-gather, as hand-written CUDA kernels.
 * Sources of the operations (cited per call below):
 *   [TACO]   "TACO: Efficient Communication Compression of Intermediate
 *            Tensors for Scalable Tensor-Parallel LLM Training" -- Core claim
 *            (data-driven reshape, Adaptive Scale-Hadamard transform,
 *            dual-scale quantization, fused compression operator), Fig. 3
 *            (FP8 E4M3), Fig. 6 / Eq. (3) (FP8 error bound), Fig. 7
 *            (overview), Fig. 9 (fused operator vs naive multi-kernel).
 *   [EQuARX] "EQuARX: Efficient Quantized AllReduce in XLA for Distributed
 *            Machine Learning Acceleration" -- What carries the argument:
 *            block-wise dynamic int8 with one FP32 scale per 64 entries,
 *            Qp1 (metadata) / Qp2 (scale data), shards converted to FP32
 *            on receipt and summed in FP32; reduce-scatter + all-gather.
 *   [FLASH]  "Flash Communication: Reducing Tensor Parallelization
 *            Bottleneck for Fast Large Language Model Inference" -- What
 *            carries the argument: asymmetric group-128 quantization, two-
 *            step All-Reduce (quantize -> All2All -> local FP32 sum ->
 *            requantize -> All-Gather -> dequantize), INT4 for the reduce
 *            stage and INT8 for the gather stage (Assumptions & free
 *            parameters).
 *
 * Conventions shared by every call:
 *  - All data pointers are DEVICE pointers (except the `shards` array of
 *    qar_reduce, which is a host array of device pointers).  The caller
 *    allocates and owns every buffer; the library never allocates, frees or
 *    synchronises.  Work is enqueued on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream) and runs asynchronously.
 *  - A tensor is `batch` independent row-major [rows, cols] matrices stacked
 *    on a leading axis.  Blocks / groups of `block` elements run along the
 *    last axis (cols % block == 0), so block k of the flat tensor covers
 *    elements [k*block, (k+1)*block) and scale k belongs to it.
 *  - Errors are returned, never raised: arguments are checked on the host
 *    before anything is enqueued (null pointers, negative sizes, shapes,
 *    16-byte alignment of x / codes / outputs, 4-byte alignment of float
 *    scales and state, 2-byte alignment of fp16 scales / zeros, unsupported
 *    scheme / block / dtype / rank count).  A launch failure returns
 *    QTA_ERR_CUDA.  An empty tensor (batch*rows*cols == 0) is a no-op that
 *    returns QTA_OK.  Kernels never trap; a pipeline wait that exceeds its
 *    time limit (about 2 s) makes the kernel stop early and record a flag
 *    that qta_device_error() reports (the stopping warp then waits at most
 *    about 2 s more for its own loads in flight, so such a kernel ends
 *    within about 4 s).
 *  - Input values must be finite; non-finite inputs give unspecified (but
 *    memory-safe) codes.
 *  - The codec calls (compress, decompress, reduce, requant, their fused
 *    forms, the ring hops, the state update and the copy) are
 *    deterministic: bit-identical results run to run.  qta_sq_error is
 *    not: the order of its FP64 partial sums is not fixed.
 */
#ifndef QTA_H
#define QTA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* qta_stream_t; /* identical to cudaStream_t */

typedef enum {
    QTA_OK = 0,
    QTA_ERR_INVALID_ARG = 1,
    QTA_ERR_ALIGNMENT = 2,
    QTA_ERR_UNSUPPORTED = 3,
    QTA_ERR_CUDA = 4
} qta_status;

typedef enum { QTA_BF16 = 0, QTA_FP16 = 1, QTA_FP32 = 2 } qta_dtype;

/* Quantization schemes and their `block`:
 *  QTA_TACO_FP8        block in {64,128,256}: block Hadamard, dual-scale
 *                      (FP32 per-tensor S + one E4M3 byte per block relative
 *                      to S), FP8 E4M3 codes with saturation at 448 [TACO].
 *  QTA_INT8_SYM_B64    block 64: int8 codes in [-127,127], one FP32 absmax
 *                      scale per block [EQuARX].
 *  QTA_INT4_ASYM_G128  block 128: 4-bit codes (element 2k in the low nibble
 *                      of byte k, 2k+1 in the high nibble), fp16 scale and
 *                      fp16 zero-point (the group minimum) per group [FLASH].
 *  QTA_INT8_ASYM_G128  block 128: as above with 8-bit codes [FLASH]. */
typedef enum {
    QTA_TACO_FP8 = 0,
    QTA_INT8_SYM_B64 = 1,
    QTA_INT4_ASYM_G128 = 2,
    QTA_INT8_ASYM_G128 = 3
} qta_scheme;

/* Per-tensor scale mode of QTA_TACO_FP8 (ignored by the INT schemes).
 *  DELAYED: use state[0] = S left by the previous step (taco_update_scale);
 *           one pass over the input, the tensor's amax is accumulated into
 *           state[1] with max().
 *  CURRENT: first compute this tensor's amax, set S = amax/448 (S = 1 if
 *           that is zero, non-finite or below FLT_MIN), state[1] = amax,
 *           then compress with it (two passes over the input).
 * ROUND_UP: a flag OR'ed into either mode.  The block scale r_b becomes
 *           the smallest E4M3 value not below a_b * t (t as in taco_compress)
 *           instead of the nearest one, so y/s_b never exceeds 448 while S
 *           covers the tensor (no saturated codes, coarser steps) -- the
 *           rounding alternative to [TACO] Fig. 7's dual scale. */
typedef enum { QTA_SCALE_DELAYED = 0, QTA_SCALE_CURRENT = 1, QTA_SCALE_ROUND_UP = 4 } qta_scale_mode;

typedef struct {
    int32_t scheme;  /* qta_scheme */
    int32_t block;   /* see qta_scheme */
    int64_t batch;   /* independent tensors, each with its own per-tensor scale */
    int64_t rows;
    int64_t cols;    /* cols % block == 0 */
    int32_t max_sms; /* SMs a call may occupy (one CTA each); 0 or >= the GPU's
                        count: all.  Leaving SMs free lets concurrent compute
                        kernels overlap the codec [FLASH: the communication
                        kernel runs on a subset of the SMs].  For calls with
                        two descriptors, the input descriptor's value counts. */
} qta_desc;

/* A quantized tensor (device pointers).
 *  codes : u8 [batch*rows*cols] (TACO, INT8 asym), i8 [..] (INT8 sym),
 *          u8 [batch*rows*cols/2] (INT4 asym)
 *  scales: u8 [n_blocks] E4M3 bits (TACO), f32 [n_blocks] (INT8 sym),
 *          fp16 bits [n_blocks] (asym)
 *  zeros : fp16 bits [n_blocks] (asym only, else unused)
 *  state : f32 [batch][2] = {S, amax} (TACO only, else unused)
 *  chan  : NULL, or (TACO only) the adaptive rescaling of the Adaptive
 *          Scale-Hadamard transform [TACO Core claim; Fig. 7: adaptive
 *          rescaling before the ASH transform]: f32 [3][cols] = down, up,
 *          amax, 16-byte aligned, shared by every tensor of a batch and by
 *          every rank of a reduction.  The compress multiplies element
 *          (row, c) by down[c] = 2^-e[c] before the transform; the decompress
 *          and the FP32 reduce multiply by up[c] = 2^e[c] after the inverse
 *          (both exact for powers of two barring underflow).  The factors
 *          come from taco_channel_amax + taco_ash_update. */
typedef struct {
    void* codes;
    void* scales;
    void* zeros;
    float* state;
    float* chan;
} qta_qtensor;

/* Byte sizes of the buffers of a quantized tensor described by `d`
 * (0 for an unused buffer or an invalid descriptor). */
size_t qta_codes_bytes(const qta_desc* d);
size_t qta_scales_bytes(const qta_desc* d);
size_t qta_zeros_bytes(const qta_desc* d);
size_t qta_state_bytes(const qta_desc* d);

/* taco_compress -- the fused compression operator [TACO Core claim, Fig. 9]
 * for every scheme: one kernel reads x once and writes codes + scales.
 * QTA_TACO_FP8: per block of `block` along the hidden axis (the reshape),
 * y = H x (unnormalised Sylvester Hadamard, butterfly strides 1,2,..,B/2 in
 * FP32), a_b = max|y|; with t = 1/(448 S) once per tensor (the product and
 * the reciprocal each rounded to FP32),
 * r_b = E4M3(a_b * t) (the product rounded to FP32, then to E4M3; raised to
 * 2^-9 if it rounds to 0 while a_b > 0), s_b = S r_b (FP32),
 * codes = E4M3_sat(y * inv) with inv = 1/s_b rounded to FP32; the amax of y
 * goes to state[1] (max-accumulated) [TACO Core claim, Fig. 7].
 * QTA_INT8_SYM_B64: a = max|x| per 64, s = a/127, q = clamp(rint(x*127/a))
 * [EQuARX Qp1/Qp2].  ASYM: s = fp16((max-min)/Q), z = fp16(min),
 * q = clamp(rint((x-z)/s), 0, Q) [FLASH].
 * x: device [batch, rows, cols] of x_dtype (bf16, fp16 or fp32), 16-byte
 * aligned.  out: buffers sized by qta_*_bytes(d); state required for TACO. */
qta_status taco_compress(const qta_desc* d, const void* x, int32_t x_dtype,
                         const qta_qtensor* out, int32_t mode, qta_stream_t stream);

/* taco_decompress -- inverse of taco_compress: dequantize in FP32; for
 * QTA_TACO_FP8 v = E4M3(q) * s_b, then the same butterfly and * (1/B); for
 * INT8 sym q*s; for asym fmaf(q, s, z); round to y_dtype (bf16 / fp16 by
 * round-to-nearest-even, or fp32) [FLASH: final dequantize of the two-step
 * All-Reduce].  y: device [batch, rows, cols], 16-byte aligned. */
qta_status taco_decompress(const qta_desc* d, const qta_qtensor* in, void* y,
                           int32_t y_dtype, qta_stream_t stream);

/* qar_reduce -- dequantize-reduce of a quantized reduce-scatter [EQuARX:
 * received shards are converted to FP32 and the partial sums kept in FP32;
 * FLASH: local FP32 sum after the All2All].  `shards` is a HOST array of
 * n_ranks quantized tensors (device buffers), each described by `d` (batch
 * must be 1), 1 <= n_ranks <= 16.  For every element of rows
 * [row_begin, row_end), in rank order: TACO / INT8 sym acc = code_0 * s_0,
 * then acc = fmaf(code_r, s_r, acc) (one FP32 rounding per rank); asym
 * acc = fmaf(q_0, s_0, z_0), then acc += fmaf(q_r, s_r, z_r).  For
 * QTA_TACO_FP8 the sum is formed in the Hadamard domain and the inverse
 * transform (butterfly, then 1/B) is applied once to it, then the channel
 * factors up[c] when the shards carry the adaptive rescaling (every shard
 * must carry the same chan pointer, else QTA_ERR_INVALID_ARG).
 * sum_out: device f32 [row_end-row_begin, cols], 16-byte aligned. */
qta_status qar_reduce(const qta_desc* d, const qta_qtensor* shards, int32_t n_ranks,
                      int64_t row_begin, int64_t row_end, float* sum_out,
                      qta_stream_t stream);

/* qar_reduce_requant -- the receiving side of one step of the two-step
 * all-reduce in one kernel: dequantize-reduce rows [row_begin, row_end) of
 * the shards and requantize the sums for the gather stage, without writing
 * an FP32 sum to memory [FLASH: local FP32 sum, then INT8 requantization
 * before the All-Gather; TACO Fig. 9: one fused operator instead of several
 * kernels].  QTA_TACO_FP8 -> QTA_TACO_FP8 with equal blocks: the sums are
 * formed in the Hadamard domain as qar_reduce forms them, and since they are
 * the transform of the reduced rows they are requantized there directly
 * (dual-scale rule of taco_compress; the inverse and forward transforms,
 * which cancel, are skipped).  Every other pair: bit-identical to qar_reduce
 * followed by qar_requant.  `d` and `shards` as for qar_reduce; `out_desc`
 * describes the requantized rows as out_desc->batch shards of out_desc->rows
 * rows each (batch * rows == row_end - row_begin, same cols), `out` its
 * buffers, `mode` its scale mode (QTA_TACO_FP8 output).  Supported scheme
 * pairs (shards -> output): TACO_FP8 -> TACO_FP8, INT8_SYM_B64 ->
 * INT8_SYM_B64, INT4_ASYM_G128 -> INT8_ASYM_G128, INT8_ASYM_G128 ->
 * INT8_ASYM_G128; other pairs return QTA_ERR_UNSUPPORTED (use the two
 * calls).  The grid is capped by d->max_sms; out_desc->max_sms is not
 * used.  With the adaptive rescaling, out->chan must be the shards' chan
 * (the factors then cancel between the reduce and the requant), else
 * QTA_ERR_UNSUPPORTED. */
qta_status qar_reduce_requant(const qta_desc* d, const qta_qtensor* shards, int32_t n_ranks,
                              int64_t row_begin, int64_t row_end, const qta_desc* out_desc,
                              const qta_qtensor* out, int32_t mode, qta_stream_t stream);

/* qar_requant -- requantization of the FP32 partial sums for the gather
 * stage [FLASH: INT8 requantization before the All-Gather; EQuARX: quantized
 * all-gather]: taco_compress with an FP32 input.  `d` describes the sum as
 * `batch` shards (each with its own per-tensor scale for TACO). */
qta_status qar_requant(const qta_desc* d, const float* sum, const qta_qtensor* out,
                       int32_t mode, qta_stream_t stream);

/* qar_dequant_add -- one hop of a quantized ring reduce-scatter at the
 * receiving rank [EQuARX What carries the argument: every received shard is
 * dequantized to FP32 before the addition; Figs. 4-5: the full-loop and
 * semi-loop adder chains are sequences of such hops].  The incoming partial
 * sum `in` (described by `d`, any batch) is dequantized exactly as
 * taco_decompress dequantizes it to FP32 (TACO: inverse butterfly, then
 * 1/B), and the receiver's own tensor x is added, one FP32 rounding per
 * element.  x: device [batch, rows, cols] of x_dtype (bf16, fp16 or fp32),
 * 16-byte aligned; sum_out: device f32 of the same shape, 16-byte aligned,
 * not overlapping x or any buffer of `in` (an overlap is detected on the
 * host and returns QTA_ERR_INVALID_ARG before anything is enqueued).
 * The ring hops take no adaptive rescaling (a chan returns
 * QTA_ERR_UNSUPPORTED).  Caller-owned buffers; errors as for the other
 * calls. */
qta_status qar_dequant_add(const qta_desc* d, const qta_qtensor* in, const void* x,
                           int32_t x_dtype, float* sum_out, qta_stream_t stream);

/* qar_dequant_add_requant -- the same hop with the partial sum requantized
 * before it travels on, in one kernel: bit-identical to qar_dequant_add
 * followed by qar_requant with `d` (same scheme, block and shape as the
 * incoming tensor; `mode` is the scale mode of a TACO output, whose state is
 * out->state).  No buffer of `out` may overlap x or a buffer of `in`
 * (checked on the host: QTA_ERR_INVALID_ARG). */
qta_status qar_dequant_add_requant(const qta_desc* d, const qta_qtensor* in, const void* x,
                                   int32_t x_dtype, const qta_qtensor* out, int32_t mode,
                                   qta_stream_t stream);

/* qta_sq_error -- *out = sum over i < n of (a_i - b_i)^2, accumulated in
 * FP64: the squared reconstruction error of a compress -> decompress round
 * trip, with which a block size is chosen per tensor [TACO Core claim:
 * data-driven reshaping -- the block size whose round trip loses least].
 * a: device [n] of a_dtype (bf16, fp16 or fp32), b: device f32 [n], both
 * 4-byte aligned; out: device double, 8-byte aligned, overwritten (the
 * order of the FP64 partial sums is not fixed: the result may differ in
 * the last bits between calls). */
qta_status qta_sq_error(const void* a, int32_t a_dtype, const float* b, int64_t n, double* out,
                        qta_stream_t stream);

/* Adaptive rescaling state: bytes of the chan buffer for `cols` channels
 * (3 * cols floats; 0 for cols <= 0).  A fresh state holds down = up = 1 and
 * amax = 0 (no rescaling). */
size_t qta_chan_bytes(int64_t cols);

/* taco_channel_amax -- per-channel statistics of the adaptive rescaling
 * [TACO Core claim: data-driven reshaping with an Adaptive Scale-Hadamard
 * transform]: chan[2*cols + c] = max(chan[2*cols + c], max over every row of
 * every tensor of |x[.., c]|).  x: device [batch, rows, cols] of x_dtype
 * (bf16, fp16, fp32), 16-byte aligned; chan: device f32 [3*cols], 16-byte
 * aligned, not overlapping x.  d gives the shape only (any valid scheme).
 * Run on the data of earlier steps (or a calibration batch); the codec calls
 * use the factors the last taco_ash_update wrote. */
qta_status taco_channel_amax(const qta_desc* d, const void* x, int32_t x_dtype, float* chan,
                             qta_stream_t stream);

/* taco_ash_update -- the channel factors from the accumulated amax, then
 * amax = 0.  Rule (the pages give none): with E(v) the binary exponent of v
 * (floor(log2 v); -127 for subnormals) and E_ref the lower median of
 * E(amax[c]) over the channels with amax[c] > 0, e[c] = min(3, max(0,
 * E(amax[c]) - E_ref - 2)) (0 for amax[c] == 0): channels at least a factor
 * 8 above the typical range are divided by up to 8.  down[c] = 2^-e[c],
 * up[c] = 2^e[c].  chan: device f32 [3*cols], 16-byte aligned.  One CTA. */
qta_status taco_ash_update(float* chan, int64_t cols, qta_stream_t stream);

/* taco_update_scale -- end-of-step update of the dual-scale state of
 * n_tensors tensors [TACO Core claim: stability across training steps]:
 * S = amax/448 (S = 1 if zero, non-finite or below FLT_MIN), amax = 0.
 * state: device f32 [n_tensors][2]. */
qta_status taco_update_scale(float* state, int64_t n_tensors, qta_stream_t stream);

/* qta_copy -- plain device-to-device copy kernel (the HBM roofline probe).
 * src, dst: device, 16-byte aligned, non-overlapping; bytes % 16 == 0. */
qta_status qta_copy(const void* src, void* dst, size_t bytes, qta_stream_t stream);

/* qta_wait_self_test -- exercises the failure path of the bounded pipeline
 * waits: a one-warp kernel waits on a shared-memory mbarrier through the
 * same wait routine every kernel uses.  complete != 0: one thread arrives
 * first and the wait succeeds at once.  complete == 0: nothing ever arrives;
 * after the wait's limit (about 2 s) the kernel records the timeout flag
 * (qta_device_error bit 0) and returns -- no trap, the context stays usable.
 * (Not an operation of the pages: a check of this library's failure
 * detection.) */
qta_status qta_wait_self_test(int32_t complete, qta_stream_t stream);

/* qta_device_error -- synchronises the current device, returns the flags
 * kernels recorded (0 = none; bit 0: a pipeline wait timed out) in *flags,
 * and clears them when `clear` is non-zero. */
qta_status qta_device_error(uint32_t* flags, int32_t clear);

/* Human-readable name of a status code (static string). */
const char* qta_status_string(qta_status s);

#ifdef __cplusplus
}
#endif
#endif /* QTA_H */
