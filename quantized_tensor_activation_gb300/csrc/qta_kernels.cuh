// qta_kernels.cuh -- the codec kernels (compress, decompress, reduce, state).
//
// Every kernel is a persistent grid of CTAs of WARPS warps.  Each warp is an
// independent streaming pipeline over "warp tiles" of 32 segments (one 64-
// element segment per lane): lane 0 keeps STAGES TMA loads in flight into a
// ring of swizzled shared-memory stages (one mbarrier each), every lane reads
// its own segment row bank-conflict free, computes in registers, and writes
// its output row into a swizzled staging buffer that lane 0 stores with one
// TMA tensor store.  No CTA-wide barrier is used after set-up, and every wait
// is bounded (see mbar_wait).
#pragma once

#include "qta_device.cuh"

namespace qta {

enum InKind : int { IN_BF16 = 0, IN_FP16 = 1, IN_FP32 = 2 };
enum SchemeKind : int { S_TACO = 0, S_INT8SYM = 1, S_ASYM4 = 2, S_ASYM8 = 3 };

// Division by a run-time invariant (Granlund-Montgomery): n / d for n < 2^31.
struct FastDiv {
    uint32_t d, m, l;
};

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f)
{
    return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(n, f.m)) + n) >> f.l);
}

// ------------------------------------------------------------ parameters
struct CompressParams {
    CUtensorMap in_map;   // 16-bit: {64, M} box {64,32} SW128; fp32: {32,2,M} box {32,1,32} SW128
    CUtensorMap out_map;  // 8-bit codes {64, M} box {64,32} SW64; 4-bit {32, M} box {32,32} SW32
    void* scales;
    void* zeros;
    float* state;
    unsigned int* err;    // device error flags (bounded waits)
    int M;                // segments
    int n_warp_tiles;     // ceil(M / 32)
    int lanes_per_block;  // block / 64 (TACO), 1 (INT8 sym), 2 (asym)
    int lanes_log2;
    FastDiv seg_per_tensor;
    int round_up;         // TACO: block scales rounded up (QTA_SCALE_ROUND_UP)
    const float* chan;    // TACO adaptive rescaling: per-channel factors down[cols] (NULL: none)
    FastDiv seg_per_row;  // cols / 64
    int chan_smem;        // the factors are copied into shared memory (cols * 4 extra bytes)
};

struct DecompressParams {
    CUtensorMap in_map;   // codes, as the compress out_map
    CUtensorMap out_map;  // 16-bit or fp32, as the compress in_map
    const void* scales;
    const void* zeros;
    const float* state;
    unsigned int* err;
    int M;
    int n_warp_tiles;
    int lanes_per_block;
    int lanes_log2;
    float inv_block;      // 1/B (TACO)
    FastDiv seg_per_tensor;
    const float* chan_up; // TACO adaptive rescaling: per-channel factors up[cols] (NULL: none)
    FastDiv seg_per_row;  // cols / 64
    int chan_smem;        // the factors are copied into shared memory (cols * 4 extra bytes)
};

struct ReduceParams {
    CUtensorMap in_map[MAX_RANKS];  // codes of each shard
    CUtensorMap out_map;            // fp32 sum {32,2,M_out}, or the requantized codes
    const void* scales[MAX_RANKS];
    const void* zeros[MAX_RANKS];
    const float* state[MAX_RANKS];
    unsigned int* err;
    int n_ranks;
    int seg_begin;                  // first input segment (row_begin * cols / 64)
    int M_out;                      // output segments
    int n_warp_tiles;
    int lanes_per_block;            // of the shards' blocks
    int lanes_log2;
    float inv_block;
    // requantization of the sum (fused reduce + requant only)
    void* q_scales;
    void* q_zeros;
    float* q_state;
    int q_lanes_per_block;
    int q_lanes_log2;
    FastDiv q_seg_per_tensor;
    int q_round_up;
    const float* chan_up; // TACO FP32 sum: per-channel factors up[cols] (NULL: none)
    FastDiv seg_per_row;  // cols / 64
    int chan_smem;        // the factors are copied into shared memory (cols * 4 extra bytes)
};

// One ring hop: the incoming quantized partial sum plus the local tensor x,
// stored as an FP32 sum or requantized with the incoming scheme and block.
struct AccumParams {
    CUtensorMap in_map;   // incoming codes, as the decompress in_map
    CUtensorMap x_map;    // local tensor, as the compress in_map
    CUtensorMap out_map;  // fp32 sum {32,2,M}, or the requantized codes
    const void* scales;
    const void* zeros;
    const float* state;
    unsigned int* err;
    int M;
    int n_warp_tiles;
    int lanes_per_block;
    int lanes_log2;
    float inv_block;
    FastDiv seg_per_tensor;
    void* q_scales;       // requantization outputs
    void* q_zeros;
    float* q_state;
    int round_up;
};

// Per-tensor amax slots of a CTA's shared-memory table (see AMAX_SLOTS).
constexpr int AMAX_SLOTS_CFG = 64;

// ------------------------------------------------------------ configuration
// Per kernel family: warps per CTA (one CTA per SM; __launch_bounds__ caps
// the registers at 64K / threads), stages of the per-warp TMA ring, and
// output staging buffers per warp.  Shared memory per CTA stays below 227 KB.
template <int IN, int SCH>
struct CompressCfg {
    static constexpr int WARPS = (IN == IN_FP32) ? 12 : 16;
    static constexpr int IN_SEG = (IN == IN_FP32) ? 256 : 128;
    static constexpr int OUT_SEG = (SCH == S_ASYM4) ? 32 : 64;
    static constexpr int STAGES = 2;
    static constexpr int IN_BYTES = 32 * IN_SEG;
    static constexpr int OUT_BYTES = 32 * OUT_SEG;
    static constexpr int OUT_BUFS = (IN == IN_FP32) ? 1 : 2;
    static constexpr int WARP_SMEM = STAGES * IN_BYTES + OUT_BUFS * OUT_BYTES;
    static constexpr int AMAX_BYTES = (SCH == S_TACO) ? 4 * AMAX_SLOTS_CFG : 0;
    static constexpr int SMEM = WARPS * WARP_SMEM + WARPS * STAGES * 8 + AMAX_BYTES + 1024;
    static constexpr int CHAN_OFF = WARPS * WARP_SMEM + WARPS * STAGES * 8 + AMAX_BYTES;   // 16-byte aligned
};

template <int SCH, int OUT>
struct DecompressCfg {
    static constexpr int WARPS = (OUT == IN_FP32) ? 12 : 16;
    static constexpr int IN_SEG = (SCH == S_ASYM4) ? 32 : 64;
    static constexpr int OUT_SEG = (OUT == IN_FP32) ? 256 : 128;
    // 2 stages: fewer loads in flight made the TACO decompress faster
    // (gpt_tp 21.3 -> 20.3 us, qwen_grad 26.6 -> 25.3 us against 4) and left
    // the INT8 ones unchanged
    static constexpr int STAGES = 2;
    static constexpr int IN_BYTES = 32 * IN_SEG;
    static constexpr int OUT_BYTES = 32 * OUT_SEG;
    static constexpr int OUT_BUFS = 1;
    static constexpr int WARP_SMEM = STAGES * IN_BYTES + OUT_BUFS * OUT_BYTES;
    static constexpr int SMEM = WARPS * WARP_SMEM + WARPS * STAGES * 8 + 1024;
    static constexpr int CHAN_OFF = WARPS * WARP_SMEM + WARPS * STAGES * 8;
};

// OSCH: OUT_F32 for the FP32 sum (qar_reduce), else the requantization scheme
// of the fused reduce + requant.
constexpr int OUT_F32 = -1;

// LG: log2 of the lanes per block of a kernel compiled for one block size, else -1.
template <int SCH, int OSCH = OUT_F32, int LG = -1>
struct ReduceCfg {
    // the INT4 kernels and the fused TACO -> TACO reduce fit 128 registers
    // and run 16 warps (the TACO one with 2-rank metadata chunks); the
    // others run 12
    static constexpr bool W16 = (SCH == S_ASYM4) || (SCH == S_TACO && OSCH == S_TACO);
    // the fused TACO reduce compiled for 4-lane blocks runs 15: on 4 x 8192 x
    // 5120 its 20480 warp tiles take 9 rounds over 152 CTAs with 16 warps or
    // 15, the last round nearly full with 15, and fewer warps share a
    // scheduler (43.1 -> 42.3 us)
    static constexpr int WARPS = (SCH == S_TACO && OSCH == S_TACO && LG == 2) ? 15 : (W16 ? 16 : 12);
    static constexpr int IN_SEG = (SCH == S_ASYM4) ? 32 : 64;
    static constexpr int OUT_SEG = (OSCH == OUT_F32) ? 256 : (OSCH == S_ASYM4) ? 32 : 64;
    // ranks whose warp tiles share one stage (one load barrier, one wait):
    // the 1 KB INT4 tiles of the fused kernel, and the TACO tiles of the fused
    // kernel compiled for 4-lane blocks, are loaded two ranks at a time
    static constexpr bool PAIRS = (SCH == S_ASYM4 && OSCH != OUT_F32) || (SCH == S_TACO && OSCH == S_TACO && LG == 2);
    static constexpr int RPU = PAIRS ? 2 : 1;
    // Stages per warp, the fastest of those measured per kernel in the step
    // (2 to 8): more stages than these put more loads in flight at once and
    // make every kernel slower.
    //   FP32 sum: INT8 2 (272 -> 250 us with 4, 8 x 16384 x 8192), TACO with
    //   1- or 2-lane blocks 3 (67.8 -> 66.6 us), INT4 and 4-lane TACO 4;
    //   fused: INT4 3 stages of two ranks (82.0 -> 79.8 us with 5), TACO 4
    //   (60.3 -> 58.1 us with 6), 4-lane TACO 2 of two ranks (42.8 -> 41.5
    //   us with 3), INT8 5 (209.3 -> 205.4 us with 8).
    static constexpr int STAGES =
        (OSCH == OUT_F32) ? ((SCH == S_INT8SYM) ? 2 : (SCH == S_TACO && LG != 2) ? 3 : 4)
                          : ((SCH == S_ASYM4) ? 6 / RPU : (W16 ? 4 / RPU : 5));
    // ranks whose scale metadata is fetched together, one chunk ahead
    static constexpr int RANK_CHUNK = (SCH == S_ASYM4) ? 8 : (W16 ? 2 : 4);
    static_assert(RANK_CHUNK % RPU == 0, "a stage never spans two metadata chunks");
    static constexpr int IN_BYTES = 32 * IN_SEG;
    // INT4 shards: a warp tile is loaded as 16 rows of two segments (64 B,
    // 64-byte swizzle) instead of 32 rows of one (on 8 x 8192 x 8192: FP32
    // sum 94.7 -> 88.1 us, fused kernel 79.8 -> 78.6 us)
    static constexpr bool ROWS64 = (SCH == S_ASYM4);
    static constexpr int STAGE_BYTES = RPU * IN_BYTES;
    static constexpr int OUT_BYTES = 32 * OUT_SEG;
    static constexpr int OUT_BUFS = 1;
    static constexpr int WARP_SMEM = STAGES * STAGE_BYTES + OUT_BUFS * OUT_BYTES;
    static constexpr int AMAX_BYTES = (OSCH == S_TACO) ? 4 * AMAX_SLOTS_CFG : 0;
    static constexpr int SMEM = WARPS * WARP_SMEM + WARPS * STAGES * 8 + AMAX_BYTES + 1024;
    static constexpr int CHAN_OFF = WARPS * WARP_SMEM + WARPS * STAGES * 8 + AMAX_BYTES;
};

// Ring hop: a stage holds a warp tile of incoming codes (2 KB slot) and of
// the local tensor (4 KB 16-bit, 8 KB fp32); OSCH as for ReduceCfg.
template <int XIN, int OSCH>
struct AccumCfg {
    static constexpr bool F32X = XIN == IN_FP32;
    static constexpr bool F32O = OSCH == OUT_F32;
    // 12 warps for the TACO and INT4 requantizing hops with a 16-bit local
    // tensor (issue-bound; 166 and 158 registers), 8 for the others
    static constexpr int WARPS = F32X ? (F32O ? 6 : 8) : ((OSCH == S_TACO || OSCH == S_ASYM4) ? 12 : 8);
    static constexpr int STAGES = 2;
    static constexpr int IN_BYTES = 32 * 64;
    static constexpr int X_BYTES = 32 * (F32X ? 256 : 128);
    static constexpr int STAGE_BYTES = IN_BYTES + X_BYTES;
    static constexpr int OUT_BYTES = 32 * (F32O ? 256 : 64);
    static constexpr int WARP_SMEM = STAGES * STAGE_BYTES + OUT_BYTES;
    static constexpr int AMAX_BYTES = (OSCH == S_TACO) ? 4 * AMAX_SLOTS_CFG : 0;
    static constexpr int SMEM = WARPS * WARP_SMEM + WARPS * STAGES * 8 + AMAX_BYTES + 1024;
};

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw)
{
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// ------------------------------------------------------------ segment I/O
// Read this lane's 64-element input segment (row `lane` of a stage) as 32
// float pairs.  xm (a multiple of 16) permutes the slots: slot j receives
// position j ^ xm (the exchange layout of fwht_cross_xl).
template <int IN>
__device__ __forceinline__ void load_segment(const uint8_t* st, int lane, u64 (&v)[32], uint32_t xm = 0)
{
    if constexpr (IN == IN_FP32) {
        const uint32_t cx = xm >> 2;   // 16-byte chunks of 4 values, 8 per box
#pragma unroll
        for (int sc = 0; sc < 16; ++sc) {
            const uint32_t pc = sc ^ cx;
            const uint4 w = lds128(st + (pc >> 3) * 4096, sw128(lane, pc & 7u));
            v[sc * 2 + 0] = pk2(__uint_as_float(w.x), __uint_as_float(w.y));
            v[sc * 2 + 1] = pk2(__uint_as_float(w.z), __uint_as_float(w.w));
        }
    } else {
        const uint32_t cx = xm >> 3;   // 16-byte chunks of 8 values
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 w = lds128(st, sw128(lane, c ^ cx));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                v[c * 4 + k] = (IN == IN_BF16) ? bf16x2_to_pair(ws[k]) : f16x2_to_pair(ws[k]);
        }
    }
}

// Write this lane's 64-element output row into a staging buffer.
template <int OUT>
__device__ __forceinline__ void store_segment(uint8_t* ob, int lane, const u64 (&v)[32])
{
    if constexpr (OUT == IN_FP32) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const u64 a = v[h * 16 + c * 2], b = v[h * 16 + c * 2 + 1];
                sts128(ob + h * 4096, sw128(lane, c), make_uint4(lo32(a), hi32(a), lo32(b), hi32(b)));
            }
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                w[k] = (OUT == IN_BF16) ? pair_to_bf16x2(v[c * 4 + k]) : pair_to_f16x2(v[c * 4 + k]);
            sts128(ob, sw128(lane, c), make_uint4(w[0], w[1], w[2], w[3]));
        }
    }
}

// Output of fwht_cross_xl into the staging rows: register group g (32/L
// pairs) goes to row (lane & ~(L-1)) + xl_group_row(g, lg, p) of the warp
// tile (p: the lane's position in its block after a swapping exchange, else
// 0), positions xm .. xm + 64/L - 1.  N4: the layout of xl_mask<true>.
template <int OUT, bool N4 = false>
__device__ __forceinline__ void store_segment_xl(uint8_t* ob, int lane, const u64 (&v)[32], int lanes_log2,
                                                 uint32_t xm, int p)
{
    const int base = lane & ~((1 << lanes_log2) - 1);
    if constexpr (OUT == IN_FP32) {
        const int kl = 4 - lanes_log2;   // log2 of the 16-byte chunks per group
#pragma unroll
        for (int sc = 0; sc < 16; ++sc) {
            const int g = sc >> kl;
            const uint32_t row = base + xl_group_row<N4>(g, lanes_log2, p);
            const uint32_t pc = (xm >> 2) + (sc & ((1 << kl) - 1));
            const u64 a = v[sc * 2], b = v[sc * 2 + 1];
            sts128(ob + (pc >> 3) * 4096, sw128(row, pc & 7u), make_uint4(lo32(a), hi32(a), lo32(b), hi32(b)));
        }
    } else {
        const int kl = 3 - lanes_log2;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int g = c >> kl;
            const uint32_t row = base + xl_group_row<N4>(g, lanes_log2, p);
            const uint32_t pc = (xm >> 3) + (c & ((1 << kl) - 1));
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                w[k] = (OUT == IN_BF16) ? pair_to_bf16x2(v[c * 4 + k]) : pair_to_f16x2(v[c * 4 + k]);
            sts128(ob, sw128(row, pc), make_uint4(w[0], w[1], w[2], w[3]));
        }
    }
}

// Byte codes of one segment from a stage (64 bytes, SW64) into 16 words;
// word group c receives the 16 codes of chunk c ^ cx.
__device__ __forceinline__ void load_codes8(const uint8_t* st, int lane, uint32_t (&q)[16], uint32_t cx = 0)
{
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 w = lds128(st, sw64(lane, c ^ cx));
        q[c * 4 + 0] = w.x;
        q[c * 4 + 1] = w.y;
        q[c * 4 + 2] = w.z;
        q[c * 4 + 3] = w.w;
    }
}

// Nibble codes of one segment (32 bytes, SW32) into 8 words.
// ROWS64: the tile as 16 rows of 64 B under the 64-byte swizzle, lane l's
// segment the half l & 1 of row l >> 1 (the 8 lanes of a wavefront still
// read 8 different 16-byte bank groups).
template <bool ROWS64 = false>
__device__ __forceinline__ void load_codes4(const uint8_t* st, int lane, uint32_t (&q)[8])
{
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint4 w = lds128(st, ROWS64 ? sw64(lane >> 1, 2 * (lane & 1) + c) : sw32(lane, c));
        q[c * 4 + 0] = w.x;
        q[c * 4 + 1] = w.y;
        q[c * 4 + 2] = w.z;
        q[c * 4 + 3] = w.w;
    }
}

// Dequantization of one segment's codes (before any transform).
// MODE 0 (assign):     TACO E4M3(q)*s, INT8 q*s
//                      ASYM fmaf(q, s, z)
// MODE 1 (accumulate): TACO/INT8 v = fmaf(code, s, v)
//                      ASYM      v = v + fmaf(q, s, z)
// INT4 takes its scale as the fp16 bits s16 (mixed-precision multiply-add);
// SC: its values come scaled by (2^-24, 2^-20) per pair (u4x8_dequant_scaled),
// and the caller scales the sum back.
// ptxas contracts a packed multiply into a packed add that consumes it in
// the same basic block.  The products of MODE 0 are only ever consumed by a
// fused multiply-add, a scalar add.rn (the first butterfly stage, which is
// never contracted), a multiply, a conversion or a store, so they keep their
// own rounding as defined.
template <int SCH, int MODE, bool SC = false, bool ROWS64 = false>
__device__ __forceinline__ void dequant_segment(const uint8_t* st, int lane, float s, float z, u64 (&v)[32],
                                                uint16_t s16, uint32_t xm = 0)
{
    const u64 s2 = pk2(s, s);
    const u64 z2 = pk2(z, z);
    // code pair c (exact) -> v[j]
    auto sym = [&](int j, u64 c) { v[j] = (MODE == 0) ? mul2(c, s2) : fma2(c, s2, v[j]); };
    auto asym = [&](int j, u64 c) {
        const u64 d = fma2(c, s2, z2);
        v[j] = (MODE == 0) ? d : add2(v[j], d);
    };
    if constexpr (SCH == S_ASYM4) {
        uint32_t q[8];
        load_codes4<ROWS64>(st, lane, q);
        auto put = [&](int w, const float (&f)[8]) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const u64 d = pk2(f[2 * k], f[2 * k + 1]);
                v[w * 4 + k] = (MODE == 0) ? d : add2(v[w * 4 + k], d);
            }
        };
        if constexpr (SC) {
            const float zlo = __fmul_rn(z, 0x1p-24f), zhi = __fmul_rn(z, 0x1p-20f);
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                float f[8];
                u4x8_dequant_scaled(q[w], s16, zlo, zhi, f);
                put(w, f);
            }
        } else {
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                float f[8];
                u4x8_dequant(q[w], s16, z, f);
                put(w, f);
            }
        }
    } else {
        uint32_t q[16];
        load_codes8(st, lane, q, xm >> 4);
#pragma unroll
        for (int w = 0; w < 16; ++w) {
            if constexpr (SCH == S_TACO) {
                sym(2 * w, e4m3x2_decode(lo16(q[w])));
                sym(2 * w + 1, e4m3x2_decode(hi16(q[w])));
            } else if constexpr (SCH == S_INT8SYM) {
                u64 a, b;
                s8x4_to_pairs(q[w], a, b);
                sym(2 * w, a);
                sym(2 * w + 1, b);
            } else {
                u64 a, b;
                u8x4_to_pairs(q[w], a, b);
                asym(2 * w, a);
                asym(2 * w + 1, b);
            }
        }
    }
}

// ------------------------------------------------------------ TMA issue
template <int IN>
__device__ __forceinline__ void issue_in16or32(const CUtensorMap* map, uint8_t* st, int row, uint64_t* bar)
{
    if constexpr (IN == IN_FP32) {
        mbar_arrive_expect_tx(bar, 8192);
        tma_load_3d(st, map, 0, 0, row, bar);
        tma_load_3d(st + 4096, map, 0, 1, row, bar);
    } else {
        mbar_arrive_expect_tx(bar, 4096);
        tma_load_2d(st, map, 0, row, bar);
    }
}

template <int OUT>
__device__ __forceinline__ void store_out16or32(const CUtensorMap* map, const uint8_t* ob, int row)
{
    if constexpr (OUT == IN_FP32) {
        tma_store_3d(map, 0, 0, row, ob);
        tma_store_3d(map, 0, 1, row, ob + 4096);
    } else {
        tma_store_2d(map, 0, row, ob);
    }
}

// ------------------------------------------------------------ adaptive rescaling
// Column of the first element of segment g (cols = 64 * spr.d per row).
__device__ __forceinline__ int seg_col0(int g, const FastDiv& spr)
{
    const uint32_t u = static_cast<uint32_t>(g);
    return static_cast<int>(u - fdiv(u, spr) * spr.d) * SEG;
}

// Multiply a lane's segment, loaded into the permuted slots of xl_mask
// (slot j holds position j ^ xm), by the per-channel factors f[col0 + position]
// (powers of two, so every product is exact barring underflow).  The products
// are consumed by scalar adds or multiplies only.
__device__ __forceinline__ void scale_slots(u64 (&v)[32], const float* __restrict__ f, int col0, uint32_t xm)
{
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const float4 c = __ldg(reinterpret_cast<const float4*>(f + col0 + ((4u * q) ^ xm)));
        v[2 * q] = mul2(v[2 * q], pk2(c.x, c.y));
        v[2 * q + 1] = mul2(v[2 * q + 1], pk2(c.z, c.w));
    }
}

// The same for values in the layout fwht_cross_xl leaves: pair j holds row
// group g = j >> (5 - lg) of the block (segment base + xl_group_row(g, lg, p),
// p = the lane's position in its block) at positions xm + 2 (j mod 2^(5-lg));
// colb is the column of the block's first element.  N4: the layout of xl_mask<true>.
template <bool N4 = false>
__device__ __forceinline__ void scale_xl(u64 (&v)[32], const float* __restrict__ f, int colb, int lg, uint32_t xm,
                                         int p)
{
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const int g = j >> (5 - lg);
        const int pos = static_cast<int>(xm) + 2 * (j & ((1 << (5 - lg)) - 1));
        const float4 c = __ldg(reinterpret_cast<const float4*>(f + colb + SEG * xl_group_row<N4>(g, lg, p) + pos));
        v[j] = mul2(v[j], pk2(c.x, c.y));
        v[j + 1] = mul2(v[j + 1], pk2(c.z, c.w));
    }
}

// The factors in shared memory: the 16-byte chunk k (4 channels) of
// segment-column j (64 channels) sits at chunk (j << 4) | (k ^ (j & 7)), so
// that the lanes of a wavefront, which read neighbouring segment-columns,
// hit different bank groups.  Every thread of the CTA copies a share, then
// the CTA synchronises.
__device__ __forceinline__ void chan_to_smem(float* fsm, const float* __restrict__ f, int cols)
{
    float4* d = reinterpret_cast<float4*>(fsm);
    const float4* g = reinterpret_cast<const float4*>(f);
    for (int i = threadIdx.x; i < cols / 4; i += blockDim.x) {
        const int j = i >> 4, k = i & 15;
        d[(j << 4) | (k ^ (j & 7))] = __ldg(g + i);
    }
    __syncthreads();
}

__device__ __forceinline__ float4 chan_sm(const float* fsm, int j, int k)
{
    return reinterpret_cast<const float4*>(fsm)[(j << 4) | (k ^ (j & 7))];
}

// scale_slots from the shared copy; j = the segment-column of the lane's segment.
__device__ __forceinline__ void scale_slots_sm(u64 (&v)[32], const float* fsm, int j, uint32_t xm)
{
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const float4 c = chan_sm(fsm, j, q ^ static_cast<int>(xm >> 2));
        v[2 * q] = mul2(v[2 * q], pk2(c.x, c.y));
        v[2 * q + 1] = mul2(v[2 * q + 1], pk2(c.z, c.w));
    }
}

// scale_xl from the shared copy; jb = the segment-column of the block's first segment.
template <bool N4 = false>
__device__ __forceinline__ void scale_xl_sm(u64 (&v)[32], const float* fsm, int jb, int lg, uint32_t xm, int p)
{
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const int g = j >> (5 - lg);
        const int pos = static_cast<int>(xm) + 2 * (j & ((1 << (5 - lg)) - 1));
        const float4 c = chan_sm(fsm, jb + xl_group_row<N4>(g, lg, p), pos >> 2);
        v[j] = mul2(v[j], pk2(c.x, c.y));
        v[j + 1] = mul2(v[j + 1], pk2(c.z, c.w));
    }
}

// ------------------------------------------------------------ quantizer
// Per-tensor amax of the dual-scale state (non-negative floats order like
// their bit patterns, so max is an unsigned atomicMax).  A CTA first gathers
// the amax of the first AMAX_SLOTS tensors in a shared-memory table and adds
// it to the global state once per tensor at its end: the warps of a fused
// reduce switch output tensor almost every tile, and one global atomic per
// tile on a handful of addresses serializes.
constexpr int AMAX_SLOTS = AMAX_SLOTS_CFG;

struct QuantOut {
    void* scales;
    void* zeros;
    float* state;
    int M;                  // segments of the quantized tensor (all batches)
    int lanes_per_block;
    int lanes_log2;
    FastDiv seg_per_tensor;
    int round_up;           // TACO block scales: smallest E4M3 value >= the ratio
    unsigned int* cta_amax; // shared-memory amax table of the CTA (TACO)
    int amax_slots;         // tensors [0, amax_slots) use the table
};

__device__ __forceinline__ void amax_add(const QuantOut& o, int tensor, uint32_t bits)
{
    if (tensor < o.amax_slots)
        atomicMax(o.cta_amax + tensor, bits);
    else
        atomicMax(reinterpret_cast<unsigned int*>(o.state + 2 * tensor + 1), bits);
}

// Zero the CTA's table (every thread calls it once, before any tile).
__device__ __forceinline__ void cta_amax_init(unsigned int* table)
{
    for (int i = threadIdx.x; i < AMAX_SLOTS; i += blockDim.x) table[i] = 0u;
    __syncthreads();
}

// Number of table slots in use for a quantized tensor of M segments.
__device__ __forceinline__ int cta_amax_slots(int M, const FastDiv& spt)
{
    const int n = static_cast<int>((static_cast<uint32_t>(M) + spt.d - 1u) / spt.d);
    return n < AMAX_SLOTS ? n : AMAX_SLOTS;
}

// Add the CTA's table to the global state (every thread calls it once, after
// its last tile and its warp's final flush).
__device__ __forceinline__ void cta_amax_flush(const unsigned int* table, float* state, int slots)
{
    __syncthreads();
    for (int i = threadIdx.x; i < slots; i += blockDim.x) {
        const unsigned int v = table[i];
        if (v != 0u) atomicMax(reinterpret_cast<unsigned int*>(state + 2 * i + 1), v);
    }
}

// Running max per warp while consecutive warp tiles stay inside one tensor,
// flushed into the table (or the global state) when the tensor changes.
struct AmaxTracker {
    int tensor = -1;
    float m = 0.0f;

    __device__ __forceinline__ void flush(const QuantOut& o, int lane)
    {
        const uint32_t w = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
        if (lane == 0 && tensor >= 0 && w != 0u) amax_add(o, tensor, w);
        m = 0.0f;
    }
};

// Drain path after a timed-out wait: let the `pending` loads this warp
// issued and has not consumed (the stages from `stage` on, in ring order)
// land before the CTA may exit.  All of them share one deadline of about
// 2 s, so a warp that gives up returns within about twice the wait limit.
__device__ __forceinline__ void drain_ring(uint64_t* bars, int stages, int stage, uint32_t phase, int pending,
                                           unsigned int* err)
{
    const uint64_t deadline = globaltimer_ns() + 2000000000ull;
    for (int i = 0; i < pending && i < stages; ++i) {
        if (!mbar_wait_until(&bars[stage], phase, deadline)) {
            atomicOr(err, ERR_WAIT_TIMEOUT);
            return;
        }
        if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

// Loads in flight for the tiles first, first + W, ... of a warp when it
// stops at tile wt: the tiles wt, wt + W, ..., wt + (stages-1) W that exist
// (each consumed tile t refilled its stage with t + stages W).
__device__ __forceinline__ int pending_tiles(int wt, int W, int n_tiles, int stages)
{
    int n = 0;
    for (int j = 0; j < stages; ++j)
        if (wt + j * W < n_tiles) ++n;
    return n;
}


// Quantizes one warp tile (one 64-element segment per lane, values in the
// original domain) into code words `ow`, writes the per-block metadata and
// accumulates the per-tensor amax (TACO).  Carries the per-warp scale cache
// and amax tracker across tiles.
template <int SCH>
struct Quantizer {
    AmaxTracker amax;
    int cached_tensor = -1;
    float S = 1.0f, tinv = 0.0f;
    // tensor of the coming tile and its scale, fetched ahead by begin()
    bool uniform = true;
    int tens = 0;
    float S_next = 1.0f;

    // Start of a warp tile: locate its tensor and fetch the per-tensor scale
    // early, so that the load has landed when run() needs it.
    __device__ __forceinline__ void begin(const QuantOut& o, int tile_first, int lane)
    {
        if constexpr (SCH == S_TACO) {
            const int g = tile_first + lane;
            const int g_last = min(tile_first + 31, o.M - 1);
            const int t_first = (int)fdiv((uint32_t)tile_first, o.seg_per_tensor);
            const int t_last = (int)fdiv((uint32_t)g_last, o.seg_per_tensor);
            uniform = (t_first == t_last);
            tens = uniform ? t_first : (int)fdiv((uint32_t)min(g, o.M - 1), o.seg_per_tensor);
            if (!uniform || tens != cached_tensor) S_next = __ldg(o.state + 2 * tens);
        }
    }

    // AMAX_ONLY: transform and record the amax, write nothing else.
    // transformed (TACO): v already holds the Hadamard-domain values.
    // XL (TACO): v holds the lane's row in the permuted slots of xl_mask, the
    // transform runs with the halved exchange, and ow comes out in its
    // layout (store_codes<..., true>); N4: the layout of xl_mask<true>.
    template <bool AMAX_ONLY, bool XL = false, bool N4 = false>
    __device__ __forceinline__ void run(u64 (&v)[32], const QuantOut& o, int tile_first, int lane,
                                        uint32_t (&ow)[16], bool transformed = false, uint32_t xm = 0)
    {
        const int g = tile_first + lane;
        const bool valid = g < o.M;
        const int L = o.lanes_per_block;
        if constexpr (SCH == S_TACO) {
            if constexpr (XL) {
                fwht64_local_xl(v, xm);
                fwht_cross_xl<false, N4>(v, L, lane);
            } else if (!transformed) {
                fwht64_local(v);
                fwht_cross(v, L, lane);
            }
            const float a = absmax64(v);
            if (uniform) {
                if (tens != amax.tensor) {
                    amax.flush(o, lane);
                    amax.tensor = tens;
                }
                amax.m = fmaxf(amax.m, a);
            } else if (valid && a > 0.0f) {
                amax_add(o, tens, __float_as_uint(a));
            }
            if constexpr (!AMAX_ONLY) {
                if (!uniform || tens != cached_tensor) {
                    S = S_next;
                    tinv = __frcp_rn(__fmul_rn(448.0f, S));
                    cached_tensor = uniform ? tens : -1;
                }
                const float ab = group_max(a, L);
                const float ratio = __fmul_rn(ab, tinv);
                uint32_t r = e4m3_encode(ratio);
                if (o.round_up && r < 0x7Eu && e4m3_decode(r) < ratio) ++r;
                if (r == 0u && ab > 0.0f) r = 1u;
                const float sb = __fmul_rn(S, e4m3_decode(r));
                const float inv = (sb > 0.0f) ? __frcp_rn(sb) : 0.0f;
                const u64 inv2 = pk2(inv, inv);
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    const float2 q0 = up2(mul2(v[2 * w], inv2));
                    const float2 q1 = up2(mul2(v[2 * w + 1], inv2));
                    ow[w] = join16(e4m3x2_encode(q0.x, q0.y), e4m3x2_encode(q1.x, q1.y));
                }
                if (valid && (lane & (L - 1)) == 0)
                    static_cast<uint8_t*>(o.scales)[g >> o.lanes_log2] = static_cast<uint8_t>(r);
            }
        } else if constexpr (SCH == S_INT8SYM) {
            const float a = absmax64(v);
            const float s = __fdiv_rn(a, 127.0f);
            float inv = (a > 0.0f) ? __fdiv_rn(127.0f, a) : 0.0f;
            if (inv > 3.40282347e+38f) inv = 0.0f;   // absmax below 127/FLT_MAX: zero codes
            const u64 inv2 = pk2(inv, inv);
            // |x * inv| <= 127.00002 < 127.5, so clamping from below at -127
            // changes no code; it also keeps the product rounded to FP32 on its
            // own before the rounding add (a fused multiply-add would round once).
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                const float2 y0 = up2(mul2(v[2 * w], inv2));
                const float2 y1 = up2(mul2(v[2 * w + 1], inv2));
                const u64 r0 = rint_bits2(pk2(fmaxf(y0.x, -127.0f), fmaxf(y0.y, -127.0f)));
                const u64 r1 = rint_bits2(pk2(fmaxf(y1.x, -127.0f), fmaxf(y1.y, -127.0f)));
                ow[w] = bytes4(lo32(r0), hi32(r0), lo32(r1), hi32(r1));
            }
            if (valid) static_cast<float*>(o.scales)[g] = s;
        } else {
            constexpr float Q = (SCH == S_ASYM4) ? 15.0f : 255.0f;
            float mn, mx;
            minmax64(v, mn, mx);
            mn = group_min(mn, 2);
            mx = group_max(mx, 2);
            float sf = __fadd_rn(__fdiv_rn(__fsub_rn(mx, mn), Q), 0.0f);
            sf = fminf(sf, 65504.0f);
            const float zc = fminf(fmaxf(__fadd_rn(mn, 0.0f), -65504.0f), 65504.0f);
            const __half s16 = __float2half_rn(sf);
            const __half z16 = __float2half_rn(zc);
            const float s = __half2float(s16), z = __half2float(z16);
            const float inv = (s > 0.0f) ? __frcp_rn(s) : 0.0f;
            const u64 inv2 = pk2(inv, inv), z2 = pk2(z, z);
            uint32_t rb[64];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float2 y = up2(mul2(sub2(v[j], z2), inv2));
                if constexpr (SCH == S_ASYM8) {
                    // round to nearest even here, clamp to [0, 255] in the pack
                    // below (flash_int4's fused reduce 79.7 -> 77.7 us against a
                    // rounding conversion to u8 and three byte permutes per word)
                    rb[2 * j] = cvt_rni_s32(y.x);
                    rb[2 * j + 1] = cvt_rni_s32(y.y);
                } else {
                    const u64 r = rint_bits2(pk2(fminf(fmaxf(y.x, 0.0f), Q), fminf(fmaxf(y.y, 0.0f), Q)));
                    rb[2 * j] = lo32(r);
                    rb[2 * j + 1] = hi32(r);
                }
            }
            if constexpr (SCH == S_ASYM4) {
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const uint32_t ev = bytes4(rb[8 * w + 0], rb[8 * w + 2], rb[8 * w + 4], rb[8 * w + 6]);
                    const uint32_t od = bytes4(rb[8 * w + 1], rb[8 * w + 3], rb[8 * w + 5], rb[8 * w + 7]);
                    ow[w] = ev | (od << 4);
                }
            } else {
#pragma unroll
                for (int w = 0; w < 16; ++w) ow[w] = pack4_sat_u8(rb[4 * w], rb[4 * w + 1], rb[4 * w + 2], rb[4 * w + 3]);
            }
            if (valid && (lane & 1) == 0) {
                static_cast<__half*>(o.scales)[g >> 1] = s16;
                static_cast<__half*>(o.zeros)[g >> 1] = z16;
            }
        }
    }

    __device__ __forceinline__ void finish(const QuantOut& o, int lane)
    {
        if constexpr (SCH == S_TACO) amax.flush(o, lane);
    }
};

// Stage one warp tile of code words in shared memory and store it with one
// TMA tensor store (8-bit codes: 64 B rows, SW64; 4-bit: 32 B rows, SW32).
// XL: ow is in the layout of fwht_cross_xl (without the row swap): word
// group g (16/L words) goes to row (lane & ~(L-1)) + xl_group_row(g, lg, 0),
// codes xm .. xm + 64/L - 1.  N4: the layout of xl_mask<true>.
template <int SCH, int OUT_BUFS, bool XL = false, bool N4 = false>
__device__ __forceinline__ void store_codes(uint8_t* ob, const CUtensorMap* map, int row, int lane,
                                            const uint32_t (&ow)[16], int lanes_log2 = 0, uint32_t xm = 0)
{
    if (lane == 0) {
        if constexpr (OUT_BUFS == 1)
            bulk_wait_read<0>();
        else
            bulk_wait_read<1>();
    }
    __syncwarp();
    if constexpr (XL) {
        const int base = lane & ~((1 << lanes_log2) - 1);
        const int kl = 2 - lanes_log2;   // log2 of the 16-byte chunks per group
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t r = base + xl_group_row<N4>(c >> kl, lanes_log2, 0);
            const uint32_t pc = (xm >> 4) + (c & ((1 << kl) - 1));
            sts128(ob, sw64(r, pc), make_uint4(ow[4 * c], ow[4 * c + 1], ow[4 * c + 2], ow[4 * c + 3]));
        }
    } else if constexpr (SCH == S_ASYM4) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
            sts128(ob, sw32(lane, c), make_uint4(ow[4 * c], ow[4 * c + 1], ow[4 * c + 2], ow[4 * c + 3]));
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            sts128(ob, sw64(lane, c), make_uint4(ow[4 * c], ow[4 * c + 1], ow[4 * c + 2], ow[4 * c + 3]));
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(map, 0, row, ob);
        bulk_commit();
    }
}

// ------------------------------------------------------------ compress
// taco_compress / qar_requant / CURRENT-mode amax pre-pass (AMAX_ONLY).
// LG: log2 of the lanes per block when fixed at compile time (TACO), else -1.
// CH: the adaptive rescaling's channel factors are applied (TACO, p.chan).
template <int IN, int SCH, bool AMAX_ONLY, int LG = -1, bool CH = false>
__global__ void __launch_bounds__(CompressCfg<IN, SCH>::WARPS * 32, 1)
compress_kernel(const __grid_constant__ CompressParams p)
{
    using C = CompressCfg<IN, SCH>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = aligned_smem(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* wb = smem + warp * C::WARP_SMEM;
    uint8_t* outb = wb + C::STAGES * C::IN_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::WARPS * C::WARP_SMEM) + warp * C::STAGES;
    unsigned int* amax_tab = reinterpret_cast<unsigned int*>(smem + C::WARPS * C::WARP_SMEM + C::WARPS * C::STAGES * 8);

    const int W = gridDim.x * C::WARPS;
    const int first = blockIdx.x * C::WARPS + warp;
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    if constexpr (SCH == S_TACO) cta_amax_init(amax_tab);
    pdl_wait();
    pdl_trigger();
    float* fsm = reinterpret_cast<float*>(smem + C::CHAN_OFF);
    if constexpr (CH)
        if (p.chan_smem) chan_to_smem(fsm, p.chan, static_cast<int>(p.seg_per_row.d) * SEG);
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            const int wt = first + s * W;
            if (wt >= p.n_warp_tiles) break;
            issue_in16or32<IN>(&p.in_map, wb + s * C::IN_BYTES, wt * 32, &bars[s]);
        }
    }
    __syncwarp();

    const int lg = (LG >= 0) ? LG : p.lanes_log2;
    const int L = 1 << lg;
    const QuantOut qo{p.scales, p.zeros, p.state, p.M, L, lg, p.seg_per_tensor,
                      p.round_up, amax_tab, (SCH == S_TACO) ? cta_amax_slots(p.M, p.seg_per_tensor) : 0};
    Quantizer<SCH> quant;
    // TACO: the rows are loaded into the permuted slots of the halved
    // cross-lane exchange
    constexpr bool XL = (SCH == S_TACO);
    // the exchange layout for 4-lane blocks when compiled for them
    constexpr bool N4 = (LG == 2);
    const uint32_t xm = XL ? xl_mask<N4>(L, lane) : 0u;
    int stage = 0;
    uint32_t phase = 0;
    int k = 0;
    bool aborted = false;
    int pending = 0;
    for (int wt = first; wt < p.n_warp_tiles; wt += W, ++k) {
        quant.begin(qo, wt * 32, lane);
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[stage], phase, p.err));
        if (!ok) {
            aborted = true;
            pending = pending_tiles(wt, W, p.n_warp_tiles, C::STAGES);
            break;
        }
        u64 v[32];
        load_segment<IN>(wb + stage * C::IN_BYTES, lane, v, xm);
        __syncwarp();
        {   // refill this stage with the tile STAGES ahead
            const int nwt = wt + C::STAGES * W;
            if (nwt < p.n_warp_tiles && lane == 0) {
                fence_proxy_async_smem();
                issue_in16or32<IN>(&p.in_map, wb + stage * C::IN_BYTES, nwt * 32, &bars[stage]);
            }
        }
        if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
        }
        // adaptive rescaling: the channel factors before the transform
        if constexpr (CH) {
            const int c0 = seg_col0(wt * 32 + lane, p.seg_per_row);
            if (p.chan_smem)
                scale_slots_sm(v, fsm, c0 / SEG, xm);
            else
                scale_slots(v, p.chan, c0, xm);
        }
        uint32_t ow[16];
        quant.template run<AMAX_ONLY, XL, N4>(v, qo, wt * 32, lane, ow, false, xm);
        if constexpr (!AMAX_ONLY)
            store_codes<SCH, C::OUT_BUFS, XL, N4>(outb + (k % C::OUT_BUFS) * C::OUT_BYTES, &p.out_map, wt * 32, lane,
                                              ow, lg, xm);
    }
    quant.finish(qo, lane);
    if (lane == 0) {
        bulk_wait_all();
        if (aborted) drain_ring(bars, C::STAGES, stage, phase, pending, p.err);
    }
    if constexpr (SCH == S_TACO) cta_amax_flush(amax_tab, p.state, qo.amax_slots);
}

// ------------------------------------------------------------ decompress
// Metadata of one segment: the dequantization scale and zero-point.
template <int SCH>
struct SegMeta {
    uint32_t raw = 0;   // TACO: scale byte; INT8: f32 bits; ASYM: s16 | z16 << 16
    float S = 0.0f;     // TACO per-tensor scale

    __device__ __forceinline__ void load(const void* scales, const void* zeros, const float* state, int g,
                                         int lanes_log2, const FastDiv& spt)
    {
        if constexpr (SCH == S_TACO) {
            raw = __ldg(static_cast<const uint8_t*>(scales) + (g >> lanes_log2));
            S = __ldg(state + 2 * (int)fdiv((uint32_t)g, spt));
        } else if constexpr (SCH == S_INT8SYM) {
            raw = __float_as_uint(__ldg(static_cast<const float*>(scales) + g));
        } else {
            const uint32_t s = __ldg(static_cast<const unsigned short*>(scales) + (g >> 1));
            const uint32_t z = __ldg(static_cast<const unsigned short*>(zeros) + (g >> 1));
            raw = s | (z << 16);
        }
    }

    __device__ __forceinline__ void decode(float& s, float& z) const
    {
        if constexpr (SCH == S_TACO) {
            s = __fmul_rn(S, e4m3_decode(raw));
            z = 0.0f;
        } else if constexpr (SCH == S_INT8SYM) {
            s = __uint_as_float(raw);
            z = 0.0f;
        } else {
            s = __half2float(__ushort_as_half(static_cast<unsigned short>(raw & 0xffffu)));
            z = __half2float(__ushort_as_half(static_cast<unsigned short>(raw >> 16)));
        }
    }
};

// LG: log2 of the lanes per block when fixed at compile time (TACO), else -1.
// CH: the adaptive rescaling's channel factors are applied (TACO, p.chan_up).
template <int SCH, int OUT, int LG = -1, bool CH = false>
__global__ void __launch_bounds__(DecompressCfg<SCH, OUT>::WARPS * 32, 1)
decompress_kernel(const __grid_constant__ DecompressParams p)
{
    using C = DecompressCfg<SCH, OUT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = aligned_smem(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* wb = smem + warp * C::WARP_SMEM;
    uint8_t* outb = wb + C::STAGES * C::IN_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::WARPS * C::WARP_SMEM) + warp * C::STAGES;
    const int W = gridDim.x * C::WARPS;
    // warp-major: the tiles of the last, partial round spread over all CTAs
    const int first = warp * gridDim.x + blockIdx.x;
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    pdl_wait();
    pdl_trigger();
    float* fsm = reinterpret_cast<float*>(smem + C::CHAN_OFF);
    if constexpr (CH)
        if (p.chan_smem) chan_to_smem(fsm, p.chan_up, static_cast<int>(p.seg_per_row.d) * SEG);
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            const int wt = first + s * W;
            if (wt >= p.n_warp_tiles) break;
            mbar_arrive_expect_tx(&bars[s], C::IN_BYTES);
            tma_load_2d(wb + s * C::IN_BYTES, &p.in_map, 0, wt * 32, &bars[s]);
        }
    }
    __syncwarp();
    const int lg = (LG >= 0) ? LG : p.lanes_log2;
    const int L = 1 << lg;
    // TACO: the codes are read into the permuted slots of the halved
    // cross-lane exchange
    // the exchange layout for 4-lane blocks when compiled for them
    constexpr bool N4 = (LG == 2);
    const uint32_t xm = (SCH == S_TACO) ? xl_mask<N4>(L, lane) : 0u;
    int stage = 0;
    uint32_t phase = 0;
    int k = 0;
    bool aborted = false;
    int pending = 0;
    // metadata of the next warp tile is fetched one tile ahead
    SegMeta<SCH> meta;
    if (first < p.n_warp_tiles && first * 32 + lane < p.M)
        meta.load(p.scales, p.zeros, p.state, first * 32 + lane, lg, p.seg_per_tensor);
    for (int wt = first; wt < p.n_warp_tiles; wt += W, ++k) {
        SegMeta<SCH> cur = meta;
        {
            const int gn = (wt + W) * 32 + lane;
            if (wt + W < p.n_warp_tiles && gn < p.M)
                meta.load(p.scales, p.zeros, p.state, gn, lg, p.seg_per_tensor);
        }
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[stage], phase, p.err));
        if (!ok) {
            aborted = true;
            pending = pending_tiles(wt, W, p.n_warp_tiles, C::STAGES);
            break;
        }
        float s, z;
        cur.decode(s, z);
        u64 v[32];
        dequant_segment<SCH, 0>(wb + stage * C::IN_BYTES, lane, s, z, v, static_cast<uint16_t>(cur.raw), xm);
        __syncwarp();
        {
            const int nwt = wt + C::STAGES * W;
            if (nwt < p.n_warp_tiles && lane == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bars[stage], C::IN_BYTES);
                tma_load_2d(wb + stage * C::IN_BYTES, &p.in_map, 0, nwt * 32, &bars[stage]);
            }
        }
        if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
        }
        if constexpr (SCH == S_TACO) {
            fwht64_local_xl(v, xm);
            fwht_cross_xl<true, N4>(v, L, lane);
            const u64 ib = pk2(p.inv_block, p.inv_block);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = mul2(v[j], ib);
            if constexpr (CH) {
                const int cb = seg_col0(wt * 32 + (lane & ~(L - 1)), p.seg_per_row);
                if (p.chan_smem)
                    scale_xl_sm<N4>(v, fsm, cb / SEG, lg, xm, lane & (L - 1));
                else
                    scale_xl<N4>(v, p.chan_up, cb, lg, xm, lane & (L - 1));
            }
        }
        uint8_t* ob = outb + (k % C::OUT_BUFS) * C::OUT_BYTES;
        if (lane == 0) {
            if constexpr (C::OUT_BUFS == 1)
                bulk_wait_read<0>();
            else
                bulk_wait_read<1>();
        }
        __syncwarp();
        if constexpr (SCH == S_TACO)
            store_segment_xl<OUT, N4>(ob, lane, v, lg, xm, lane & (L - 1));
        else
            store_segment<OUT>(ob, lane, v);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            store_out16or32<OUT>(&p.out_map, ob, wt * 32);
            bulk_commit();
        }
    }
    if (lane == 0) {
        bulk_wait_all();
        if (aborted) drain_ring(bars, C::STAGES, stage, phase, pending, p.err);
    }
}

// ------------------------------------------------------------ reduce
// Units of the stage ring are (warp tile, rank) pairs, rank fastest; the
// issuing lane walks them with a cursor (tile index t, rank r).
struct UnitCursor {
    int t = 0, r = 0;
    __device__ __forceinline__ void advance(int n_ranks, int ranks_per_unit = 1)
    {
        r += ranks_per_unit;
        if (r >= n_ranks) {
            r = 0;
            ++t;
        }
    }
};

template <int SCH, int OSCH, int LG>
__device__ __forceinline__ void reduce_issue(const ReduceParams& p, uint8_t* wb, uint64_t* bars,
                                             int stage, const UnitCursor& u, int first, int W, int n)
{
    using C = ReduceCfg<SCH, OSCH, LG>;
    const int wt = first + u.t * W;
    const int nr = min(C::RPU, n - u.r);
    mbar_arrive_expect_tx(&bars[stage], nr * C::IN_BYTES);
#pragma unroll
    for (int i = 0; i < C::RPU; ++i)
        if (i < nr)
            tma_load_2d(wb + stage * C::STAGE_BYTES + i * C::IN_BYTES, &p.in_map[u.r + i], 0,
                        C::ROWS64 ? (p.seg_begin + wt * 32) >> 1 : p.seg_begin + wt * 32, &bars[stage]);
}

// Ranks are processed in chunks of RANK_CHUNK; the scale metadata of the next
// chunk is fetched while the current one is accumulated (TACO: the block
// scale bytes; the shards' per-tensor scales are read from the CTA's shared
// copy when a rank is decoded).
template <int SCH, int RANK_CHUNK>
__device__ __forceinline__ void reduce_meta_load(const ReduceParams& p, int t, int c, int first, int W, int lane,
                                                 int n, SegMeta<SCH> (&m)[RANK_CHUNK])
{
    const int o = (first + t * W) * 32 + lane;
    const int g = p.seg_begin + o;
    const bool valid = o < p.M_out;
#pragma unroll
    for (int k = 0; k < RANK_CHUNK; ++k) {
        const int r = c * RANK_CHUNK + k;
        if (valid && r < n) {
            if constexpr (SCH == S_TACO) {
                m[k].raw = __ldg(static_cast<const uint8_t*>(p.scales[r]) + (g >> p.lanes_log2));
            } else if constexpr (SCH == S_INT8SYM) {
                m[k].raw = __float_as_uint(__ldg(static_cast<const float*>(p.scales[r]) + g));
            } else {
                const uint32_t s = __ldg(static_cast<const unsigned short*>(p.scales[r]) + (g >> 1));
                const uint32_t z = __ldg(static_cast<const unsigned short*>(p.zeros[r]) + (g >> 1));
                m[k].raw = s | (z << 16);
            }
        } else {
            m[k].raw = 0u;
            m[k].S = 0.0f;
        }
    }
}

// qar_reduce (OSCH = OUT_F32) and the fused qar_reduce_requant (OSCH = the
// requantization scheme; AMAX_ONLY = its CURRENT-mode pre-pass).  The sum of
// a warp tile is formed exactly as qar_reduce forms it and then quantized
// exactly as qar_requant quantizes an FP32 input -- bit-identical to the two
// calls -- except for TACO -> TACO with equal blocks, where the Hadamard-
// domain sum is requantized directly.
// LG: log2 of the shards' lanes per block when fixed at compile time (the
// TACO FP32 sum, which inverts the transform with the halved exchange), else -1.
// CH: the adaptive rescaling's channel factors are applied to the TACO FP32
// sum (p.chan_up).
// NR: the number of shards when compiled in (> 0; it must equal p.n_ranks),
// else 0.  With it the rank loop unrolls completely, and the shard of every
// metadata load and TMA load is a constant.
template <int SCH, int OSCH, bool AMAX_ONLY, int LG = -1, bool CH = false, int NR = 0>
__global__ void __launch_bounds__(ReduceCfg<SCH, OSCH, LG>::WARPS * 32, 1)
reduce_kernel(const __grid_constant__ ReduceParams p)
{
    using C = ReduceCfg<SCH, OSCH, LG>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = aligned_smem(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* wb = smem + warp * C::WARP_SMEM;
    uint8_t* outb = wb + C::STAGES * C::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::WARPS * C::WARP_SMEM) + warp * C::STAGES;
    unsigned int* amax_tab = reinterpret_cast<unsigned int*>(smem + C::WARPS * C::WARP_SMEM + C::WARPS * C::STAGES * 8);
    const int W = gridDim.x * C::WARPS;
    // warp-major: the tiles of the last, partial round spread over all CTAs
    const int first = warp * gridDim.x + blockIdx.x;
    const int n = NR > 0 ? NR : p.n_ranks;
    const int my_tiles = (first < p.n_warp_tiles) ? (p.n_warp_tiles - first + W - 1) / W : 0;
    const int total_units = my_tiles * ((n + C::RPU - 1) / C::RPU);
    UnitCursor next_unit;   // next unit to load (meaningful in lane 0)
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    if constexpr (OSCH == S_TACO) cta_amax_init(amax_tab);
    pdl_wait();
    pdl_trigger();
    // per-tensor scales of the shards, read once per CTA
    __shared__ float sS[MAX_RANKS];
    if constexpr (SCH == S_TACO) {
        if (threadIdx.x < p.n_ranks) sS[threadIdx.x] = __ldg(p.state[threadIdx.x]);
        __syncthreads();
    }
    float* fsm = reinterpret_cast<float*>(smem + C::CHAN_OFF);
    if constexpr (CH)
        if (p.chan_smem) chan_to_smem(fsm, p.chan_up, static_cast<int>(p.seg_per_row.d) * SEG);
    if (lane == 0) {
        for (int u = 0; u < C::STAGES && u < total_units; ++u) {
            reduce_issue<SCH, OSCH, LG>(p, wb, bars, u, next_unit, first, W, n);
            next_unit.advance(n, C::RPU);
        }
    }
    __syncwarp();
    const int L = (LG >= 0) ? (1 << LG) : p.lanes_per_block;
    // TACO FP32 sum: codes read into the permuted slots of the halved exchange
    constexpr bool XL = (SCH == S_TACO) && (OSCH == OUT_F32);
    // the exchange layout for 4-lane blocks when compiled for them
    constexpr bool N4 = (LG == 2);
    const uint32_t xm = XL ? xl_mask<N4>(L, lane) : 0u;
    constexpr int RANK_CHUNK = C::RANK_CHUNK;
    const int n_chunks = (n + RANK_CHUNK - 1) / RANK_CHUNK;
    constexpr int CHUNKS_NR = NR > 0 ? (NR + RANK_CHUNK - 1) / RANK_CHUNK : 1;
    // INT4: the rank terms and partial sums are formed scaled by powers of two
    // (no nibble subtraction) and the sum is scaled back after the last rank
    constexpr bool SCALED4 = SCH == S_ASYM4;
    int stage = 0;
    uint32_t phase = 0;
    int unit = 0;
    bool aborted = false;
    // TACO -> TACO compiled for one block size: the output's lanes equal the input's
    constexpr bool SAME_LG = (LG >= 0) && (SCH == S_TACO) && (OSCH == S_TACO);
    const QuantOut qo{p.q_scales, p.q_zeros, p.q_state, p.M_out, SAME_LG ? L : p.q_lanes_per_block,
                      SAME_LG ? LG : p.q_lanes_log2, p.q_seg_per_tensor, p.q_round_up, amax_tab,
                      (OSCH == S_TACO) ? cta_amax_slots(p.M_out, p.q_seg_per_tensor) : 0};
    Quantizer<(OSCH == OUT_F32) ? S_TACO : OSCH> quant;
    SegMeta<SCH> nxt[RANK_CHUNK];
    if (my_tiles > 0) reduce_meta_load<SCH, RANK_CHUNK>(p, 0, 0, first, W, lane, n, nxt);
    for (int t = 0; t < my_tiles && !aborted; ++t) {
        const int wt = first + t * W;
        if constexpr (OSCH != OUT_F32) quant.begin(qo, wt * 32, lane);
        u64 acc[32];
        auto chunk = [&](int c) {
            SegMeta<SCH> cur[RANK_CHUNK];
#pragma unroll
            for (int kk = 0; kk < RANK_CHUNK; ++kk) cur[kk] = nxt[kk];
            if (c + 1 < n_chunks)
                reduce_meta_load<SCH, RANK_CHUNK>(p, t, c + 1, first, W, lane, n, nxt);
            else if (t + 1 < my_tiles)
                reduce_meta_load<SCH, RANK_CHUNK>(p, t + 1, 0, first, W, lane, n, nxt);
#pragma unroll
            for (int kk = 0; kk < RANK_CHUNK; ++kk) {
                const int r = c * RANK_CHUNK + kk;
                if (r >= n) break;
                const int slot = kk % C::RPU;   // this rank's tile within the stage
                if (slot == 0) {
                    const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[stage], phase, p.err));
                    if (!ok) {
                        aborted = true;
                        break;
                    }
                }
                float s, z;
                if constexpr (SCH == S_TACO) {
                    s = __fmul_rn(sS[r], e4m3_decode(cur[kk].raw));
                    z = 0.0f;
                } else {
                    cur[kk].decode(s, z);
                }
                const uint16_t s16 = static_cast<uint16_t>(cur[kk].raw);
                const uint8_t* tile = wb + stage * C::STAGE_BYTES + slot * C::IN_BYTES;
                if (r == 0)
                    dequant_segment<SCH, 0, SCALED4, C::ROWS64>(tile, lane, s, z, acc, s16, xm);
                else
                    dequant_segment<SCH, 1, SCALED4, C::ROWS64>(tile, lane, s, z, acc, s16, xm);
                if (slot == C::RPU - 1 || r == n - 1) {
                    __syncwarp();
                    if constexpr (NR > 0) {
                        // the unit STAGES ahead of this one: with the rank count
                        // compiled in, its tile offset and shard are constants
                        constexpr int U = (NR + C::RPU - 1) / C::RPU;
                        const int ahead = (c * RANK_CHUNK + kk) / C::RPU + C::STAGES;
                        const UnitCursor u{t + ahead / U, (ahead % U) * C::RPU};
                        if (lane == 0 && u.t < my_tiles) {
                            fence_proxy_async_smem();
                            reduce_issue<SCH, OSCH, LG>(p, wb, bars, stage, u, first, W, n);
                        }
                    } else if (lane == 0 && unit + C::STAGES < total_units) {
                        fence_proxy_async_smem();
                        reduce_issue<SCH, OSCH, LG>(p, wb, bars, stage, next_unit, first, W, n);
                        next_unit.advance(n, C::RPU);
                    }
                    ++unit;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        };
        if constexpr (NR > 0) {
#pragma unroll
            for (int c = 0; c < CHUNKS_NR; ++c)
                if (!aborted) chunk(c);
        } else {
            for (int c = 0; c < n_chunks && !aborted; ++c) chunk(c);
        }
        if (aborted) break;
        if constexpr (SCALED4) {
            // the INT4 sums back from their (2^-24, 2^-20) scales (exact)
            const u64 un = pk2(0x1p24f, 0x1p20f);
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = mul2(acc[j], un);
        }
        // TACO -> TACO with equal blocks: the sums already are the Hadamard
        // transform of the reduced rows, so they are requantized as they are
        // (the inverse and forward transforms cancel and are skipped).
        const bool direct = SAME_LG || ((SCH == S_TACO) && (OSCH == S_TACO) && (p.q_lanes_per_block == L));
        if (SCH == S_TACO && !direct) {
            if constexpr (XL) {
                fwht64_local_xl(acc, xm);
                fwht_cross_xl<false, N4>(acc, L, lane);
            } else {
                fwht64_local(acc);
                fwht_cross(acc, L, lane);
            }
            if constexpr (OSCH == OUT_F32) {
                const u64 ib = pk2(p.inv_block, p.inv_block);
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[j] = mul2(acc[j], ib);
                if constexpr (CH && XL) {
                    const int cb = seg_col0(p.seg_begin + wt * 32 + (lane & ~(L - 1)), p.seg_per_row);
                    if (p.chan_smem)
                        scale_xl_sm<N4>(acc, fsm, cb / SEG, (LG >= 0) ? LG : p.lanes_log2, xm, 0);
                    else
                        scale_xl<N4>(acc, p.chan_up, cb, (LG >= 0) ? LG : p.lanes_log2, xm, 0);
                }
            } else {
                // scalar rounded multiplies: the requantizer's butterfly adds
                // follow, and a packed multiply would be contracted into them
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float2 t2 = up2(acc[j]);
                    acc[j] = pk2(__fmul_rn(t2.x, p.inv_block), __fmul_rn(t2.y, p.inv_block));
                }
            }
        }
        if constexpr (OSCH == OUT_F32) {
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            if constexpr (XL)
                store_segment_xl<IN_FP32, N4>(outb, lane, acc, (LG >= 0) ? LG : p.lanes_log2, xm, 0);
            else
                store_segment<IN_FP32>(outb, lane, acc);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                store_out16or32<IN_FP32>(&p.out_map, outb, wt * 32);
                bulk_commit();
            }
        } else {
            uint32_t ow[16];
            quant.template run<AMAX_ONLY>(acc, qo, wt * 32, lane, ow, direct);
            if constexpr (!AMAX_ONLY) store_codes<OSCH, 1>(outb, &p.out_map, wt * 32, lane, ow);
        }
    }
    if constexpr (OSCH != OUT_F32) quant.finish(qo, lane);
    if (lane == 0) {
        bulk_wait_all();
        // units [unit, unit + STAGES) that exist were issued and not consumed
        if (aborted) drain_ring(bars, C::STAGES, stage, phase, min(C::STAGES, total_units - unit), p.err);
    }
    if constexpr (OSCH == S_TACO) cta_amax_flush(amax_tab, p.q_state, qo.amax_slots);
}

// ------------------------------------------------------------ ring hop
// v[j] = v[j] * (1/B) (TACO) + x[j], one rounding each, with x read chunk
// by chunk from this lane's row of the stage.  The multiply is packed and
// the add scalar: ptxas contracts a packed multiply only into a packed add.
template <int SCH, int XIN>
__device__ __forceinline__ void add_local_segment(const uint8_t* st, int lane, u64 (&v)[32], float inv_block)
{
    const u64 ib2 = pk2(inv_block, inv_block);
    auto add = [&](int j, float bx, float by) {
        const float2 a = up2((SCH == S_TACO) ? mul2(v[j], ib2) : v[j]);
        v[j] = pk2(__fadd_rn(a.x, bx), __fadd_rn(a.y, by));
    };
    if constexpr (XIN == IN_FP32) {
#pragma unroll
        for (int sc = 0; sc < 16; ++sc) {
            const uint4 w = lds128(st + (sc >> 3) * 4096, sw128(lane, sc & 7));
            add(sc * 2, __uint_as_float(w.x), __uint_as_float(w.y));
            add(sc * 2 + 1, __uint_as_float(w.z), __uint_as_float(w.w));
        }
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 w = lds128(st, sw128(lane, c));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 b = up2((XIN == IN_BF16) ? bf16x2_to_pair(ws[k]) : f16x2_to_pair(ws[k]));
                add(c * 4 + k, b.x, b.y);
            }
        }
    }
}

// qar_dequant_add (OSCH = OUT_F32) and qar_dequant_add_requant (OSCH = SCH;
// AMAX_ONLY = its CURRENT-mode pre-pass): the incoming codes are dequantized
// exactly as taco_decompress dequantizes them to FP32 (TACO: inverse
// butterfly, then 1/B), the local tensor is added with one scalar FP32
// rounding per element, and the sum is stored, or quantized exactly as
// qar_requant quantizes an FP32 input.  LG: log2 of the lanes per block when
// fixed at compile time (TACO), else -1.
template <int SCH, int XIN, int OSCH, bool AMAX_ONLY, int LG = -1>
__global__ void __launch_bounds__(AccumCfg<XIN, OSCH>::WARPS * 32, 1)
accum_kernel(const __grid_constant__ AccumParams p)
{
    using C = AccumCfg<XIN, OSCH>;
    constexpr int CODE_BYTES = 32 * ((SCH == S_ASYM4) ? 32 : 64);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = aligned_smem(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* wb = smem + warp * C::WARP_SMEM;
    uint8_t* outb = wb + C::STAGES * C::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::WARPS * C::WARP_SMEM) + warp * C::STAGES;
    unsigned int* amax_tab = reinterpret_cast<unsigned int*>(smem + C::WARPS * C::WARP_SMEM + C::WARPS * C::STAGES * 8);
    const int W = gridDim.x * C::WARPS;
    const int first = blockIdx.x * C::WARPS + warp;
    auto issue = [&](int s, int wt) {
        uint8_t* st = wb + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&bars[s], CODE_BYTES + C::X_BYTES);
        tma_load_2d(st, &p.in_map, 0, wt * 32, &bars[s]);
        if constexpr (XIN == IN_FP32) {
            tma_load_3d(st + C::IN_BYTES, &p.x_map, 0, 0, wt * 32, &bars[s]);
            tma_load_3d(st + C::IN_BYTES + 4096, &p.x_map, 0, 1, wt * 32, &bars[s]);
        } else {
            tma_load_2d(st + C::IN_BYTES, &p.x_map, 0, wt * 32, &bars[s]);
        }
    };
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    if constexpr (OSCH == S_TACO) cta_amax_init(amax_tab);
    pdl_wait();
    pdl_trigger();
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            const int wt = first + s * W;
            if (wt >= p.n_warp_tiles) break;
            issue(s, wt);
        }
    }
    __syncwarp();
    const int lg = (LG >= 0) ? LG : p.lanes_log2;
    const int L = 1 << lg;
    const QuantOut qo{p.q_scales, p.q_zeros, p.q_state, p.M, L, lg, p.seg_per_tensor,
                      p.round_up, amax_tab, (OSCH == S_TACO) ? cta_amax_slots(p.M, p.seg_per_tensor) : 0};
    Quantizer<(OSCH == OUT_F32) ? S_TACO : OSCH> quant;
    int stage = 0;
    uint32_t phase = 0;
    bool aborted = false;
    int pending = 0;
    SegMeta<SCH> meta;   // metadata of the next warp tile, fetched one tile ahead
    if (first < p.n_warp_tiles && first * 32 + lane < p.M)
        meta.load(p.scales, p.zeros, p.state, first * 32 + lane, p.lanes_log2, p.seg_per_tensor);
    for (int wt = first; wt < p.n_warp_tiles; wt += W) {
        SegMeta<SCH> cur = meta;
        {
            const int gn = (wt + W) * 32 + lane;
            if (wt + W < p.n_warp_tiles && gn < p.M)
                meta.load(p.scales, p.zeros, p.state, gn, p.lanes_log2, p.seg_per_tensor);
        }
        if constexpr (OSCH != OUT_F32) quant.begin(qo, wt * 32, lane);
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[stage], phase, p.err));
        if (!ok) {
            aborted = true;
            pending = pending_tiles(wt, W, p.n_warp_tiles, C::STAGES);
            break;
        }
        float s, z;
        cur.decode(s, z);
        u64 v[32];
        const uint8_t* st = wb + stage * C::STAGE_BYTES;
        dequant_segment<SCH, 0>(st, lane, s, z, v, static_cast<uint16_t>(cur.raw));
        if constexpr (SCH == S_TACO) {
            fwht64_local(v);
            fwht_cross(v, L, lane);
        }
        // times 1/B (TACO), then the local tensor with one rounding per
        // element: scalar rounded operations, which are never contracted.
        // The local tensor is read from the stage a 16-byte chunk at a time.
        add_local_segment<SCH, XIN>(st + C::IN_BYTES, lane, v, p.inv_block);
        __syncwarp();
        {
            const int nwt = wt + C::STAGES * W;
            if (nwt < p.n_warp_tiles && lane == 0) {
                fence_proxy_async_smem();
                issue(stage, nwt);
            }
        }
        if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
        }
        if constexpr (OSCH == OUT_F32) {
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            store_segment<IN_FP32>(outb, lane, v);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                store_out16or32<IN_FP32>(&p.out_map, outb, wt * 32);
                bulk_commit();
            }
        } else {
            uint32_t ow[16];
            quant.template run<AMAX_ONLY>(v, qo, wt * 32, lane, ow);
            if constexpr (!AMAX_ONLY) store_codes<OSCH, 1>(outb, &p.out_map, wt * 32, lane, ow);
        }
    }
    if constexpr (OSCH != OUT_F32) quant.finish(qo, lane);
    if (lane == 0) {
        bulk_wait_all();
        if (aborted) drain_ring(bars, C::STAGES, stage, phase, pending, p.err);
    }
    if constexpr (OSCH == S_TACO) cta_amax_flush(amax_tab, p.q_state, qo.amax_slots);
}

// ------------------------------------------------------------ small kernels
enum StateOp : int { STATE_UPDATE = 0, STATE_RESET_AMAX = 1, STATE_SET_SCALE = 2 };

__global__ void state_kernel(float* state, long long n, int op);
__global__ void copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long n16);
cudaError_t launch_channel_amax(const void* x, int kind, long long n_rows, long long cols, float* amax,
                                cudaStream_t stream);
cudaError_t launch_ash_update(float* chan, long long cols, cudaStream_t stream);

}  // namespace qta
