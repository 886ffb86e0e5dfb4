/*
 * qta_oracle.h -- plain, slow, single-threaded CPU oracle of the quantized
 * tensor-activation codec.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the benchmark's CPU-baseline leg may call it; the product path
 * (the CUDA library) never does, and the two share no code or headers.
 *
 * Sources (each function cites the passage it follows):
 *   [TACO]   "TACO: Efficient Communication Compression of Intermediate
 *            Tensors for Scalable Tensor-Parallel LLM Training" (review page):
 *            Core claim; Fig. 3 (E4M3 vs E5M2); Fig. 6 / Eq. (3) (FP8 ULP
 *            bound); Fig. 7 (overview: rescaling, ASH transform, dual-scale);
 *            Fig. 8 (distribution before/after the Hadamard rotation).
 *   [EQuARX] "EQuARX: Efficient Quantized AllReduce in XLA for Distributed
 *            Machine Learning Acceleration" (review page): What carries the
 *            argument (block-wise int8, one FP32 scale per 64 entries,
 *            Qp1/Qp2, dequantize to FP32 before adding).
 *            Figs. 4-5 (full-loop / semi-loop adder chains of the ring).
 *   [FLASH]  "Flash Communication: Reducing Tensor Parallelization Bottleneck
 *            for Fast Large Language Model Inference" (review page): What
 *            carries the argument (asymmetric group-128 quantization, two-step
 *            All-Reduce, INT4 reduce / INT8 gather), Assumptions & free
 *            parameters (group size 128, bit widths).
 *
 * Layouts (all row-major, blocks are contiguous along the last axis):
 *   x       [batch][rows][cols]  bf16 / fp16 / fp32
 *   TACO    codes u8 [batch*rows*cols]   (E4M3 bits)
 *           scales u8 [batch*rows*cols/B] (E4M3 bits, relative to S)
 *           state f32 [batch][2] = {S, amax}
 *   INT8    codes i8 [..cols], scales f32 [..cols/64]
 *   ASYM b  codes u8 [..cols*b/8] (b=4: element 2k low nibble, 2k+1 high),
 *           scales f16 bits [..cols/128], zeros f16 bits [..cols/128]
 */
#ifndef QTA_ORACLE_H
#define QTA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BF16 = 0, ORC_FP16 = 1, ORC_FP32 = 2 };
enum { ORC_TACO_FP8 = 0, ORC_INT8_SYM = 1, ORC_INT4_ASYM = 2, ORC_INT8_ASYM = 3 };
enum { ORC_DELAYED = 0, ORC_CURRENT = 1, ORC_ROUND_UP = 4 };

/* ---- number formats ---- */
uint8_t  orc_e4m3_encode(float v);
float    orc_e4m3_decode(uint8_t c);
uint16_t orc_f32_to_bf16(float v);
uint16_t orc_f32_to_f16(float v);
float    orc_bf16_to_f32(uint16_t h);
float    orc_f16_to_f32(uint16_t h);
void     orc_e4m3_encode_array(const float* v, uint8_t* out, int64_t n);
void     orc_f32_to_bf16_array(const float* v, uint16_t* out, int64_t n);
void     orc_f32_to_f16_array(const float* v, uint16_t* out, int64_t n);

/* ---- block Hadamard ---- */
void orc_fwht(float* y, int B);               /* in place, unnormalised */
void orc_fwht_rows(float* y, int64_t nblk, int B);

/* ---- per-tensor scale rule and update ---- */
float orc_scale_from_amax(float amax);
void  orc_taco_update_scale(float* state, int64_t batch);

/* ---- compress / decompress ---- */
int orc_compress(int scheme, int B, const void* x, int in_dtype, int64_t batch,
                 int64_t rows, int64_t cols, float* state, int mode,
                 void* codes, void* scales, void* zeros);
int orc_decompress(int scheme, int B, const void* codes, const void* scales,
                   const void* zeros, const float* state, int64_t batch,
                   int64_t rows, int64_t cols, void* y, int out_dtype);

/* ---- dequantize-reduce over n_ranks shards, rows [row_begin,row_end) ---- */
int orc_reduce(int scheme, int B, int n_ranks, const void* const* codes,
               const void* const* scales, const void* const* zeros,
               const float* const* states, int64_t rows, int64_t cols,
               int64_t row_begin, int64_t row_end, float* sum_out);

/* ---- fused dequantize-reduce + requantize ---- */
int orc_reduce_requant(int scheme, int B, int n_ranks, const void* const* codes,
                       const void* const* scales, const void* const* zeros,
                       const float* const* states, int64_t rows, int64_t cols,
                       int64_t row_begin, int64_t row_end, int out_scheme, int out_B,
                       int64_t out_batch, float* out_state, int mode, void* out_codes,
                       void* out_scales, void* out_zeros);

/* ---- ring hop: dequantize the incoming partial sum, add the local tensor ---- */
int orc_dequant_add(int scheme, int B, const void* codes, const void* scales, const void* zeros,
                    const float* state, int64_t batch, int64_t rows, int64_t cols, const void* x,
                    int x_dtype, float* sum_out);

/* ---- adaptive rescaling (per-channel powers of two); chan = float[3*cols]:
 *      down[cols], up[cols], amax[cols] ---- */
int orc_channel_amax(const void* x, int dtype, int64_t batch, int64_t rows, int64_t cols, float* chan);
int orc_ash_update(float* chan, int64_t cols);
int orc_compress_chan(int scheme, int B, const void* x, int in_dtype, int64_t batch,
                      int64_t rows, int64_t cols, float* state, int mode,
                      void* codes, void* scales, void* zeros, const float* chan);
int orc_decompress_chan(int scheme, int B, const void* codes, const void* scales,
                        const void* zeros, const float* state, int64_t batch,
                        int64_t rows, int64_t cols, void* y, int out_dtype, const float* chan);
int orc_reduce_chan(int scheme, int B, int n_ranks, const void* const* codes,
                    const void* const* scales, const void* const* zeros,
                    const float* const* states, int64_t rows, int64_t cols,
                    int64_t row_begin, int64_t row_end, float* sum_out, const float* chan);
int orc_reduce_requant_chan(int scheme, int B, int n_ranks, const void* const* codes,
                            const void* const* scales, const void* const* zeros,
                            const float* const* states, int64_t rows, int64_t cols,
                            int64_t row_begin, int64_t row_end, int out_scheme, int out_B,
                            int64_t out_batch, float* out_state, int mode, void* out_codes,
                            void* out_scales, void* out_zeros, const float* chan);

#ifdef __cplusplus
}
#endif
#endif
