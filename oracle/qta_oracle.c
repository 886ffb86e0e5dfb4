/*
 * qta_oracle.c -- the CPU oracle.  TEST INFRASTRUCTURE ONLY (see the header):
 * plain scalar C, one thread, no blocking or fusion beyond what each method
 * states, built with -O2 -ffp-contract=off -fno-fast-math so that every
 * float operation below is one IEEE-754 binary32 operation rounded to
 * nearest-even, in the order written.
 *
 * The pages fix FP32 as the working precision of the method (EQuARX: shards
 * are dequantized to FP32 and summed in FP32; TACO: FP32 per-tensor scale),
 * so the oracle computes in binary32; every integer it produces (a code, a
 * scale byte) is decided in that precision.  Where the pages leave a step
 * open, the plainest reading that the rest supports is taken; each is stated
 * where it is used, marked "Reading".
 */
#include "qta_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* Round the non-negative integer sig * 2^-shift to the nearest integer,
 * ties to even (reading: every rounding is round-to-nearest-even). */
static uint32_t rne_shift(uint32_t sig, int shift)
{
    if (shift <= 0) return sig << (-shift);
    if (shift >= 32) return 0; /* sig < 2^24 < half of 2^shift */
    uint32_t q = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return q;
}

/* ------------------------------------------------------------------------
 * FP8 E4M3 (the "E4M3" of [TACO] Fig. 3; the FN variant of the FP8 paper the
 * TACO page cites: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, 0x7F/0xFF = NaN, largest finite 448, subnormal step 2^-9).
 * ---------------------------------------------------------------------- */
float orc_e4m3_decode(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    float mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexpf((float)m, -9);            /* m/8 * 2^-6 */
    else
        mag = ldexpf((float)(8 + m), e - 10);  /* (1+m/8) * 2^(e-7) */
    return s ? -mag : mag;
}

/* Encode with round-to-nearest-even onto the E4M3 grid; magnitudes that
 * round above 448 saturate to 448, +-Inf -> +-448,
 * NaN -> 0x7F.  The sign of zero is kept. */
uint8_t orc_e4m3_encode(float v)
{
    uint32_t u = f2u(v);
    uint8_t sign = (uint8_t)((u >> 31) << 7);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return 0x7f;
    if (a == 0x7f800000u) return sign | 0x7e;
    int ef = (int)(a >> 23);
    if (ef == 0) return sign; /* binary32 subnormals are < 2^-126: round to 0 */
    int E = ef - 127;                         /* |v| in [2^E, 2^(E+1)) */
    uint32_t sig = (a & 0x7fffffu) | 0x800000u; /* |v| = sig * 2^(E-23) */
    int k = (E < -6 ? -6 : E) - 3;            /* grid step: 2^k */
    uint32_t n = rne_shift(sig, 23 + k - E);  /* |v| / 2^k rounded */
    uint32_t code;
    if (E < -6)
        code = n;                             /* subnormal: n steps of 2^-9 */
    else
        code = (uint32_t)((E + 7) << 3) + n - 8u; /* n in [8,16] */
    if (code > 0x7eu) code = 0x7eu;           /* satfinite */
    return sign | (uint8_t)code;
}

void orc_e4m3_encode_array(const float* v, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

/* ------------------------------------------------------------------------
 * bf16 / fp16 (IEEE binary16), round-to-nearest-even, overflow to +-Inf
 * (the standard conversion), NaN to a quiet NaN.
 * ---------------------------------------------------------------------- */
float orc_bf16_to_f32(uint16_t h) { return u2f((uint32_t)h << 16); }

uint16_t orc_f32_to_bf16(float v)
{
    uint32_t u = f2u(v);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t q = u >> 16, rem = u & 0xffffu;
    if (rem > 0x8000u || (rem == 0x8000u && (q & 1u))) q += 1u; /* carries into exp */
    return (uint16_t)q;
}

float orc_f16_to_f32(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    float mag;
    if (e == 31) mag = m ? NAN : INFINITY;
    else if (e == 0) mag = ldexpf((float)m, -24);
    else mag = ldexpf((float)(1024 + m), e - 25);
    return s ? -mag : mag;
}

uint16_t orc_f32_to_f16(float v)
{
    uint32_t u = f2u(v);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return sign | 0x7e00u;
    if (a == 0x7f800000u) return sign | 0x7c00u;
    int ef = (int)(a >> 23);
    if (ef == 0) return sign;
    int E = ef - 127;
    uint32_t sig = (a & 0x7fffffu) | 0x800000u;
    if (E > 15) return sign | 0x7c00u;
    int k = (E < -14 ? -14 : E) - 10;
    uint32_t n = rne_shift(sig, 23 + k - E);
    uint32_t code = (E < -14) ? n : (uint32_t)((E + 15) << 10) + n - 1024u;
    if (code >= 0x7c00u) code = 0x7c00u;     /* rounded past 65504 -> Inf */
    return sign | (uint16_t)code;
}

void orc_f32_to_bf16_array(const float* v, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(v[i]);
}

void orc_f32_to_f16_array(const float* v, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(v[i]);
}

static float load_elem(const void* x, int dtype, int64_t i)
{
    if (dtype == ORC_BF16) return orc_bf16_to_f32(((const uint16_t*)x)[i]);
    if (dtype == ORC_FP16) return orc_f16_to_f32(((const uint16_t*)x)[i]);
    return ((const float*)x)[i];
}

static void store_elem(void* y, int dtype, int64_t i, float v)
{
    if (dtype == ORC_BF16) ((uint16_t*)y)[i] = orc_f32_to_bf16(v);
    else if (dtype == ORC_FP16) ((uint16_t*)y)[i] = orc_f32_to_f16(v);
    else ((float*)y)[i] = v;
}

/* ------------------------------------------------------------------------
 * Block Hadamard ([TACO] Core claim, Fig. 7, Fig. 8: the Hadamard rotation
 * of the Adaptive Scale-Hadamard transform).  Reading: unnormalised Sylvester
 * matrix, H[i][j] = (-1)^popcount(i & j), applied as the in-place butterfly
 * with strides h = 1, 2, 4, ..., B/2 in that order; each pair (j, j+h) with
 * j & h == 0 becomes (a + b, a - b) in binary32.
 * ---------------------------------------------------------------------- */
void orc_fwht(float* y, int B)
{
    for (int h = 1; h < B; h <<= 1)
        for (int i = 0; i < B; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = y[j], b = y[j + h];
                y[j] = a + b;
                y[j + h] = a - b;
            }
}

void orc_fwht_rows(float* y, int64_t nblk, int B)
{
    for (int64_t b = 0; b < nblk; ++b) orc_fwht(y + b * B, B);
}

/* ------------------------------------------------------------------------
 * Per-tensor FP32 scale of the dual-scale scheme ([TACO] Core claim:
 * dual-scale quantization keeps FP8 stable across training steps).
 * Reading: S = amax / 448 from the latest amax (history length one); a zero,
 * non-finite or sub-normal result falls back to S = 1.
 * ---------------------------------------------------------------------- */
float orc_scale_from_amax(float amax)
{
    float S = amax / 448.0f;
    if (!(S >= FLT_MIN && S <= FLT_MAX)) S = 1.0f;
    return S;
}

void orc_taco_update_scale(float* state, int64_t batch)
{
    for (int64_t t = 0; t < batch; ++t) {
        state[2 * t] = orc_scale_from_amax(state[2 * t + 1]);
        state[2 * t + 1] = 0.0f;
    }
}

/* ---- TACO FP8 compress of one tensor ([TACO] Core claim, Fig. 7) ----
 * Reading: blocks are B contiguous elements along the hidden (last) axis.
 * Reading: block scale r_b = E4M3(a_b / (448 S)) stored as one E4M3 byte relative
 *     to the per-tensor FP32 scale S; s_b = S * r_b; codes E4M3(y * 1/s_b). */
/* Dual-scale FP8 quantization of nblk transformed blocks y (block scale and
 * per-tensor scale as read above). */
/* mode: ORC_DELAYED or ORC_CURRENT, optionally OR'ed with ORC_ROUND_UP: the
 * block scale r_b is then the smallest E4M3 value not below a_b / (448 S)
 * instead of the nearest one, so that y / s_b stays within 448 whenever S
 * covers the tensor (no saturated codes: the rounding alternative to the
 * nearest block scale of [TACO] Fig. 7's dual scale). */
static void taco_quantize_blocks(const float* y, int64_t nblk, int B, float* st, int mode,
                                 uint8_t* codes, uint8_t* scales)
{
    const int round_up = (mode & ORC_ROUND_UP) != 0;
    mode &= ~ORC_ROUND_UP;
    if (mode == ORC_CURRENT) {
        float amax = 0.0f;
        for (int64_t i = 0; i < nblk * B; ++i) amax = fmaxf(amax, fabsf(y[i]));
        st[0] = orc_scale_from_amax(amax);
        st[1] = 0.0f;
    }
    float S = st[0];
    float tinv = 1.0f / (448.0f * S);
    float amax_t = 0.0f;
    for (int64_t b = 0; b < nblk; ++b) {
        const float* yb = y + b * B;
        float a = 0.0f;
        for (int i = 0; i < B; ++i) a = fmaxf(a, fabsf(yb[i]));
        amax_t = fmaxf(amax_t, a);
        const float ratio = a * tinv;
        uint8_t r = orc_e4m3_encode(ratio);
        if (round_up && r < 0x7E && orc_e4m3_decode(r) < ratio) r = (uint8_t)(r + 1);
        if (r == 0 && a > 0.0f) r = 0x01;
        float sb = S * orc_e4m3_decode(r);
        float inv = (sb > 0.0f) ? 1.0f / sb : 0.0f;
        for (int i = 0; i < B; ++i) codes[b * B + i] = orc_e4m3_encode(yb[i] * inv);
        scales[b] = r;
    }
    st[1] = fmaxf(st[1], amax_t);
}

/* ---- TACO FP8 compress of one tensor ([TACO] Core claim, Fig. 7):
 * the adaptive rescaling (when `down` is given: element i of a row, channel
 * c = i mod cols, is multiplied by the power of two down[c] in FP32), the
 * block Hadamard of every block, then the dual-scale quantization. */
static int taco_compress_tensor(const void* x, int dtype, int64_t off, int64_t E, int64_t cols, int B,
                                const float* down, float* st, int mode, uint8_t* codes, uint8_t* scales)
{
    float* y = (float*)malloc(sizeof(float) * (size_t)(E > 0 ? E : 1));
    if (!y) return -2;
    for (int64_t i = 0; i < E; ++i) {
        y[i] = load_elem(x, dtype, off + i);
        if (down) y[i] = y[i] * down[i % cols];
    }
    orc_fwht_rows(y, E / B, B);
    taco_quantize_blocks(y, E / B, B, st, mode, codes, scales);
    free(y);
    return 0;
}

/* ---- block-symmetric INT8, one FP32 scale per 64 ([EQuARX] What carries
 * the argument: Qp1 computes the absmax metadata, Qp2 scales the data).
 * Reading: the 64 entries of one scale are 64 contiguous elements. */
static void int8sym_compress_tensor(const void* x, int dtype, int64_t off, int64_t E,
                                    int8_t* codes, float* scales)
{
    for (int64_t b = 0; b < E / 64; ++b) {
        float a = 0.0f;
        for (int i = 0; i < 64; ++i) a = fmaxf(a, fabsf(load_elem(x, dtype, off + b * 64 + i)));
        float s = a / 127.0f;
        float inv = (a > 0.0f) ? 127.0f / a : 0.0f;
        if (inv > FLT_MAX) inv = 0.0f; /* a < 127/FLT_MAX: the block is stored as zeros */
        for (int i = 0; i < 64; ++i) {
            float q = rintf(load_elem(x, dtype, off + b * 64 + i) * inv);
            if (q > 127.0f) q = 127.0f;
            if (q < -127.0f) q = -127.0f;
            codes[b * 64 + i] = (int8_t)q;
        }
        scales[b] = s;
    }
}

/* ---- asymmetric group-128 INT4 / INT8 ([FLASH] What carries the argument,
 * Assumptions & free parameters: g = 128, fp16 scale + zero-point per group).
 * Reading: min/max affine quantizer with a floating zero-point equal to the group
 * minimum: s = fp16((max-min)/Q), z = fp16(min), q = clamp(rint((x-z)/s)).
 * Reading: INT4 codes, element 2k in the low nibble of byte k, 2k+1 in the high. */
static void asym_compress_tensor(const void* x, int dtype, int64_t off, int64_t E,
                                 int bits, uint8_t* codes, uint16_t* scales,
                                 uint16_t* zeros)
{
    const int G = 128;
    const float Q = (float)((1 << bits) - 1);
    for (int64_t g = 0; g < E / G; ++g) {
        float mn = load_elem(x, dtype, off + g * G), mx = mn;
        for (int i = 1; i < G; ++i) {
            float v = load_elem(x, dtype, off + g * G + i);
            mn = fminf(mn, v);
            mx = fmaxf(mx, v);
        }
        /* "+ 0.0f" stores a zero scale / zero-point as +0, so that which of
         * -0 and +0 a min / max picks (an order detail) cannot show. */
        float sf = (mx - mn) / Q + 0.0f;
        if (sf > 65504.0f) sf = 65504.0f;
        float zc = mn + 0.0f;
        if (zc > 65504.0f) zc = 65504.0f;
        if (zc < -65504.0f) zc = -65504.0f;
        uint16_t s16 = orc_f32_to_f16(sf), z16 = orc_f32_to_f16(zc);
        float s = orc_f16_to_f32(s16), z = orc_f16_to_f32(z16);
        float inv = (s > 0.0f) ? 1.0f / s : 0.0f;
        for (int i = 0; i < G; ++i) {
            float q = rintf((load_elem(x, dtype, off + g * G + i) - z) * inv);
            if (q < 0.0f) q = 0.0f;
            if (q > Q) q = Q;
            uint8_t c = (uint8_t)q;
            int64_t e = g * G + i;
            if (bits == 8) {
                codes[e] = c;
            } else if ((e & 1) == 0) {
                codes[e >> 1] = c;
            } else {
                codes[e >> 1] = (uint8_t)(codes[e >> 1] | (c << 4));
            }
        }
        scales[g] = s16;
        zeros[g] = z16;
    }
}

static int check_shape(int scheme, int B, int64_t batch, int64_t rows, int64_t cols)
{
    if (batch < 0 || rows < 0 || cols < 0) return -1;
    if (scheme == ORC_TACO_FP8) {
        if (B < 2 || (B & (B - 1)) || B > 4096) return -1;
    } else if (scheme == ORC_INT8_SYM) {
        if (B != 64) return -1;
    } else if (scheme == ORC_INT4_ASYM || scheme == ORC_INT8_ASYM) {
        if (B != 128) return -1;
    } else {
        return -1;
    }
    if (cols % B) return -1;
    return 0;
}

int orc_compress_chan(int scheme, int B, const void* x, int in_dtype, int64_t batch,
                      int64_t rows, int64_t cols, float* state, int mode,
                      void* codes, void* scales, void* zeros, const float* chan)
{
    if (check_shape(scheme, B, batch, rows, cols)) return -1;
    if (chan && scheme != ORC_TACO_FP8) return -1;
    int64_t E = rows * cols;
    if (scheme == ORC_TACO_FP8) {
        for (int64_t t = 0; t < batch; ++t)
            if (taco_compress_tensor(x, in_dtype, t * E, E, cols, B, chan, state + 2 * t, mode,
                                     (uint8_t*)codes + t * E, (uint8_t*)scales + t * (E / B)))
                return -2;
    } else if (scheme == ORC_INT8_SYM) {
        for (int64_t t = 0; t < batch; ++t)
            int8sym_compress_tensor(x, in_dtype, t * E, E, (int8_t*)codes + t * E,
                                    (float*)scales + t * (E / 64));
    } else {
        int bits = scheme == ORC_INT4_ASYM ? 4 : 8;
        for (int64_t t = 0; t < batch; ++t)
            asym_compress_tensor(x, in_dtype, t * E, E, bits,
                                 (uint8_t*)codes + t * (E * bits / 8),
                                 (uint16_t*)scales + t * (E / 128), (uint16_t*)zeros + t * (E / 128));
    }
    return 0;
}

int orc_compress(int scheme, int B, const void* x, int in_dtype, int64_t batch,
                 int64_t rows, int64_t cols, float* state, int mode,
                 void* codes, void* scales, void* zeros)
{
    return orc_compress_chan(scheme, B, x, in_dtype, batch, rows, cols, state, mode, codes, scales, zeros, 0);
}

/* The decoded code (exact) and the FP32 dequantization scale of element e
 * for the symmetric schemes: TACO E4M3(q) and s_b = S * r_b; INT8 q and s. */
static void code_and_scale(int scheme, int B, const void* codes, const void* scales, const float* st,
                           int64_t e, float* code, float* sc)
{
    if (scheme == ORC_TACO_FP8) {
        *sc = st[0] * orc_e4m3_decode(((const uint8_t*)scales)[e / B]);
        *code = orc_e4m3_decode(((const uint8_t*)codes)[e]);
    } else {
        *sc = ((const float*)scales)[e / 64];
        *code = (float)((const int8_t*)codes)[e];
    }
}

/* Dequantized value of element e (flat index within one tensor) in FP32.
 * TACO: E4M3 code times s_b = S * r_b, before the inverse transform.
 * INT8: q * s.  ASYM: fmaf(q, s, z) (one rounding, the asymmetric reading above). */
static float dequant(int scheme, int B, const void* codes, const void* scales,
                     const void* zeros, const float* st, int64_t e)
{
    if (scheme == ORC_TACO_FP8) {
        float sb = st[0] * orc_e4m3_decode(((const uint8_t*)scales)[e / B]);
        return orc_e4m3_decode(((const uint8_t*)codes)[e]) * sb;
    }
    if (scheme == ORC_INT8_SYM)
        return (float)((const int8_t*)codes)[e] * ((const float*)scales)[e / 64];
    float s = orc_f16_to_f32(((const uint16_t*)scales)[e / 128]);
    float z = orc_f16_to_f32(((const uint16_t*)zeros)[e / 128]);
    int q;
    if (scheme == ORC_INT8_ASYM)
        q = ((const uint8_t*)codes)[e];
    else
        q = (((const uint8_t*)codes)[e >> 1] >> ((e & 1) * 4)) & 15;
    return fmaf((float)q, s, z);
}

/* Decompress: dequantize; for TACO apply the inverse Hadamard (the same
 * butterfly, then times 1/B, an exact power of two), then, with the
 * adaptive rescaling, times the channel's power of two up[c] (the inverse of
 * the compress's down[c]); round to out dtype. */
int orc_decompress_chan(int scheme, int B, const void* codes, const void* scales,
                        const void* zeros, const float* state, int64_t batch,
                        int64_t rows, int64_t cols, void* y, int out_dtype, const float* chan)
{
    if (check_shape(scheme, B, batch, rows, cols)) return -1;
    if (chan && scheme != ORC_TACO_FP8) return -1;
    const float* up = chan ? chan + cols : 0;
    int64_t E = rows * cols;
    float* v = (float*)malloc(sizeof(float) * (size_t)B);
    if (!v) return -2;
    for (int64_t t = 0; t < batch; ++t) {
        const uint8_t* c8 = (const uint8_t*)codes;
        const void* ct;
        const void* sc;
        const void* zt = 0;
        if (scheme == ORC_TACO_FP8) {
            ct = c8 + t * E;
            sc = (const uint8_t*)scales + t * (E / B);
        } else if (scheme == ORC_INT8_SYM) {
            ct = c8 + t * E;
            sc = (const float*)scales + t * (E / 64);
        } else {
            int bits = scheme == ORC_INT4_ASYM ? 4 : 8;
            ct = c8 + t * (E * bits / 8);
            sc = (const uint16_t*)scales + t * (E / 128);
            zt = (const uint16_t*)zeros + t * (E / 128);
        }
        const float* st = state ? state + 2 * t : 0;
        for (int64_t b = 0; b < E / B; ++b) {
            for (int i = 0; i < B; ++i) v[i] = dequant(scheme, B, ct, sc, zt, st, b * B + i);
            if (scheme == ORC_TACO_FP8) {
                orc_fwht(v, B);
                for (int i = 0; i < B; ++i) v[i] = v[i] * (1.0f / (float)B);
                if (up)
                    for (int i = 0; i < B; ++i) v[i] = v[i] * up[(b * B + i) % cols];
            }
            for (int i = 0; i < B; ++i) store_elem(y, out_dtype, t * E + b * B + i, v[i]);
        }
    }
    free(v);
    return 0;
}

int orc_decompress(int scheme, int B, const void* codes, const void* scales,
                   const void* zeros, const float* state, int64_t batch,
                   int64_t rows, int64_t cols, void* y, int out_dtype)
{
    return orc_decompress_chan(scheme, B, codes, scales, zeros, state, batch, rows, cols, y, out_dtype, 0);
}

/* Dequantize-reduce ([EQuARX] What carries the argument: each received shard
 * is converted to FP32 first and the partial sums are kept in FP32;
 * [FLASH] What carries the argument: local FP32 sum after the All2All).
 * Reading: per element, in rank order r = 0 .. N-1, with the dequantized term in
 * FP32 arithmetic entering the FP32 partial sum:
 *   TACO, INT8:  acc = code_0 * s_0;  acc = fmaf(code_r, s_r, acc)
 *                (the product code * scale is exact inside the fused
 *                multiply-add; one FP32 rounding per rank)
 *   ASYM:        acc = fmaf(q_0, s_0, z_0);  acc = acc + fmaf(q_r, s_r, z_r)
 * TACO sums in the Hadamard domain and applies the inverse transform once to
 * the sum (then 1/B). */
/* The per-element sums of rows [row_begin, row_end) before any transform
 * (the rank-order reading above), written to acc. */
static void reduce_sums(int scheme, int B, int n_ranks, const void* const* codes,
                        const void* const* scales, const void* const* zeros,
                        const float* const* states, int64_t cols, int64_t row_begin,
                        int64_t row_end, float* acc_out)
{
    int64_t e0 = row_begin * cols, e1 = row_end * cols;
    for (int64_t e = e0; e < e1; ++e) {
        float acc = 0.0f;
        for (int r = 0; r < n_ranks; ++r) {
            const void* z = zeros ? zeros[r] : 0;
            const float* st = states ? states[r] : 0;
            if (r == 0) {
                acc = dequant(scheme, B, codes[r], scales[r], z, st, e);
            } else if (scheme == ORC_TACO_FP8 || scheme == ORC_INT8_SYM) {
                float code, sc;
                code_and_scale(scheme, B, codes[r], scales[r], st, e, &code, &sc);
                acc = fmaf(code, sc, acc);
            } else {
                acc = acc + dequant(scheme, B, codes[r], scales[r], z, st, e);
            }
        }
        acc_out[e - e0] = acc;
    }
}

/* With the adaptive rescaling (chan given, the same for every rank: the
 * ranks' pre-scaled tensors then sum to the pre-scaled sum, whose transform
 * is the sum of their transforms), the sum is multiplied by up[c] after the
 * inverse transform, as the decompress does. */
int orc_reduce_chan(int scheme, int B, int n_ranks, const void* const* codes,
                    const void* const* scales, const void* const* zeros,
                    const float* const* states, int64_t rows, int64_t cols,
                    int64_t row_begin, int64_t row_end, float* sum_out, const float* chan)
{
    if (check_shape(scheme, B, 1, rows, cols)) return -1;
    if (n_ranks < 1 || row_begin < 0 || row_end < row_begin || row_end > rows) return -1;
    if (chan && scheme != ORC_TACO_FP8) return -1;
    reduce_sums(scheme, B, n_ranks, codes, scales, zeros, states, cols, row_begin, row_end, sum_out);
    if (scheme == ORC_TACO_FP8) {
        int64_t n = (row_end - row_begin) * cols;
        for (int64_t b0 = 0; b0 < n; b0 += B) {
            orc_fwht(sum_out + b0, B);
            for (int i = 0; i < B; ++i) sum_out[b0 + i] = sum_out[b0 + i] * (1.0f / (float)B);
            if (chan)
                for (int i = 0; i < B; ++i) sum_out[b0 + i] = sum_out[b0 + i] * chan[cols + (b0 + i) % cols];
        }
    }
    return 0;
}

int orc_reduce(int scheme, int B, int n_ranks, const void* const* codes,
               const void* const* scales, const void* const* zeros,
               const float* const* states, int64_t rows, int64_t cols,
               int64_t row_begin, int64_t row_end, float* sum_out)
{
    return orc_reduce_chan(scheme, B, n_ranks, codes, scales, zeros, states, rows, cols, row_begin, row_end,
                           sum_out, 0);
}

/* Fused dequantize-reduce + requantize of rows [row_begin, row_end) into
 * out_batch output tensors of (row_end-row_begin)/out_batch rows each.
 * TACO -> TACO with equal blocks: the sums are already in the Hadamard
 * domain of the output blocks -- they are the transform of the reduced rows
 * -- so they are requantized there directly (the inverse and the forward
 * transform, which cancel, are not applied).  Every other pair: qar_reduce
 * then the compress of its FP32 rows. */
/* chan (adaptive rescaling, TACO -> TACO only): the shards' and the
 * output's channel factors, one set.  Equal blocks: the Hadamard-domain
 * sums are the transform of the pre-scaled reduced rows and are requantized
 * as they are; otherwise the reduce (times up[c]) then the compress (times
 * down[c]). */
int orc_reduce_requant_chan(int scheme, int B, int n_ranks, const void* const* codes,
                            const void* const* scales, const void* const* zeros,
                            const float* const* states, int64_t rows, int64_t cols,
                            int64_t row_begin, int64_t row_end, int out_scheme, int out_B,
                            int64_t out_batch, float* out_state, int mode, void* out_codes,
                            void* out_scales, void* out_zeros, const float* chan)
{
    if (check_shape(scheme, B, 1, rows, cols)) return -1;
    if (chan && (scheme != ORC_TACO_FP8 || out_scheme != ORC_TACO_FP8)) return -1;
    if (n_ranks < 1 || row_begin < 0 || row_end < row_begin || row_end > rows) return -1;
    int64_t nrows = row_end - row_begin;
    if (out_batch < 1 || nrows % out_batch) return -1;
    if (check_shape(out_scheme, out_B, out_batch, nrows / out_batch, cols)) return -1;
    float* acc = (float*)malloc(sizeof(float) * (size_t)(nrows * cols > 0 ? nrows * cols : 1));
    if (!acc) return -2;
    int rc = 0;
    if (scheme == ORC_TACO_FP8 && out_scheme == ORC_TACO_FP8 && B == out_B) {
        reduce_sums(scheme, B, n_ranks, codes, scales, zeros, states, cols, row_begin, row_end, acc);
        int64_t Et = nrows / out_batch * cols;
        for (int64_t t = 0; t < out_batch; ++t)
            taco_quantize_blocks(acc + t * Et, Et / B, B, out_state + 2 * t, mode,
                                 (uint8_t*)out_codes + t * Et, (uint8_t*)out_scales + t * (Et / B));
    } else {
        rc = orc_reduce_chan(scheme, B, n_ranks, codes, scales, zeros, states, rows, cols, row_begin,
                             row_end, acc, chan);
        if (!rc)
            rc = orc_compress_chan(out_scheme, out_B, acc, ORC_FP32, out_batch, nrows / out_batch, cols,
                                   out_state, mode, out_codes, out_scales, out_zeros, chan);
    }
    free(acc);
    return rc;
}

int orc_reduce_requant(int scheme, int B, int n_ranks, const void* const* codes,
                       const void* const* scales, const void* const* zeros,
                       const float* const* states, int64_t rows, int64_t cols,
                       int64_t row_begin, int64_t row_end, int out_scheme, int out_B,
                       int64_t out_batch, float* out_state, int mode, void* out_codes,
                       void* out_scales, void* out_zeros)
{
    return orc_reduce_requant_chan(scheme, B, n_ranks, codes, scales, zeros, states, rows, cols, row_begin,
                                   row_end, out_scheme, out_B, out_batch, out_state, mode, out_codes,
                                   out_scales, out_zeros, 0);
}

/* One hop of a ring reduce-scatter [EQuARX] What carries the argument (each
 * received shard is dequantized to FP32 before it is added; the partial sum
 * is requantized before it travels on) and Figs. 4-5 (full-loop and
 * semi-loop adder chains): the incoming quantized partial sum is dequantized
 * to FP32 exactly as orc_decompress does it (TACO: inverse transform, then
 * 1/B), and the receiver's own tensor x (bf16, fp16 or fp32) is added with
 * one FP32 rounding per element.  sum_out: f32 [batch, rows, cols]. */
int orc_dequant_add(int scheme, int B, const void* codes, const void* scales, const void* zeros,
                    const float* state, int64_t batch, int64_t rows, int64_t cols, const void* x,
                    int x_dtype, float* sum_out)
{
    int rc = orc_decompress(scheme, B, codes, scales, zeros, state, batch, rows, cols, sum_out, ORC_FP32);
    if (rc) return rc;
    int64_t n = batch * rows * cols;
    for (int64_t e = 0; e < n; ++e) sum_out[e] = sum_out[e] + load_elem(x, x_dtype, e);
    return 0;
}

/* ------------------------------------------------------------------------
 * Adaptive rescaling of the Adaptive Scale-Hadamard transform ([TACO] Core
 * claim: data-driven reshaping together with an Adaptive Scale-Hadamard
 * transform; Fig. 7: tensors are compressed via adaptive rescaling, the ASH
 * transform and dual-scale quantization).  The pages give no rule.
 * Reading: every hidden channel c gets a power of two down[c] = 2^-e[c]
 * that multiplies the channel before the block Hadamard (and up[c] = 2^e[c]
 * after the inverse), shared by all ranks of a reduction, so that channels
 * far above the typical channel range no longer dominate the Hadamard
 * blocks they fall in.  The exponents come from the per-channel amax of
 * earlier data (caller-owned state, like the per-tensor scale):
 *   E(v)  = floor(log2 v) for a normal v > 0 (its binary exponent), -127 for
 *           a subnormal v;
 *   E_ref = the lower median of E(amax[c]) over the channels with amax > 0;
 *   e[c]  = min(3, max(0, E(amax[c]) - E_ref - 2)), 0 when amax[c] == 0:
 *           channels less than a factor 8 above the typical range keep
 *           factor 1; larger ones are divided by up to 8, which leaves
 *           them at about four times the typical range.  (On the outlier-
 *           channel workloads this rule lowered the round-trip error most
 *           robustly among the thresholds and caps tried; a larger cap
 *           amplifies the error of rare extreme channels.)
 * chan = float[3 * cols]: down[cols], up[cols], amax[cols].
 * ---------------------------------------------------------------------- */
int orc_channel_amax(const void* x, int dtype, int64_t batch, int64_t rows, int64_t cols, float* chan)
{
    if (batch < 0 || rows < 0 || cols <= 0) return -1;
    float* amax = chan + 2 * cols;
    for (int64_t r = 0; r < batch * rows; ++r)
        for (int64_t c = 0; c < cols; ++c) amax[c] = fmaxf(amax[c], fabsf(load_elem(x, dtype, r * cols + c)));
    return 0;
}

static int binary_exponent(float v)
{
    uint32_t u = f2u(v) & 0x7fffffffu;
    int ef = (int)(u >> 23);
    return ef == 0 ? -127 : ef - 127;
}

static int cmp_int(const void* a, const void* b)
{
    int x = *(const int*)a, y = *(const int*)b;
    return (x > y) - (x < y);
}

int orc_ash_update(float* chan, int64_t cols)
{
    if (cols <= 0) return -1;
    float* down = chan;
    float* up = chan + cols;
    float* amax = chan + 2 * cols;
    int* ex = (int*)malloc(sizeof(int) * (size_t)cols);
    if (!ex) return -2;
    int64_t n = 0;
    for (int64_t c = 0; c < cols; ++c)
        if (amax[c] > 0.0f) ex[n++] = binary_exponent(amax[c]);
    qsort(ex, (size_t)n, sizeof(int), cmp_int);
    int e_ref = n > 0 ? ex[(n - 1) / 2] : 0;
    free(ex);
    for (int64_t c = 0; c < cols; ++c) {
        int e = 0;
        if (amax[c] > 0.0f) {
            e = binary_exponent(amax[c]) - e_ref - 2;
            if (e < 0) e = 0;
            if (e > 3) e = 3;
        }
        down[c] = ldexpf(1.0f, -e);
        up[c] = ldexpf(1.0f, e);
        amax[c] = 0.0f;
    }
    return 0;
}
