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
};

struct ReduceParams {
    CUtensorMap in_map[MAX_RANKS];  // codes of each shard
    CUtensorMap out_map;            // fp32 {32,2,M_out}
    const void* scales[MAX_RANKS];
    const void* zeros[MAX_RANKS];
    const float* state[MAX_RANKS];
    unsigned int* err;
    int n_ranks;
    int seg_begin;                  // first input segment (row_begin * cols / 64)
    int M_out;                      // output segments
    int n_warp_tiles;
    int lanes_per_block;
    int lanes_log2;
    float inv_block;
};

// ------------------------------------------------------------ configuration
template <int IN, int SCH>
struct CompressCfg {
    static constexpr int WARPS = 8;
    static constexpr int IN_SEG = (IN == IN_FP32) ? 256 : 128;
    static constexpr int OUT_SEG = (SCH == S_ASYM4) ? 32 : 64;
    static constexpr int STAGES = (IN == IN_FP32) ? 2 : 4;
    static constexpr int IN_BYTES = 32 * IN_SEG;
    static constexpr int OUT_BYTES = 32 * OUT_SEG;
    static constexpr int OUT_BUFS = 2;
    static constexpr int WARP_SMEM = STAGES * IN_BYTES + OUT_BUFS * OUT_BYTES;
    static constexpr int SMEM = WARPS * WARP_SMEM + WARPS * STAGES * 8 + 1024;
};

template <int SCH, int OUT>
struct DecompressCfg {
    static constexpr int WARPS = 8;
    static constexpr int IN_SEG = (SCH == S_ASYM4) ? 32 : 64;
    static constexpr int OUT_SEG = (OUT == IN_FP32) ? 256 : 128;
    static constexpr int STAGES = 6;
    static constexpr int IN_BYTES = 32 * IN_SEG;
    static constexpr int OUT_BYTES = 32 * OUT_SEG;
    static constexpr int OUT_BUFS = 2;
    static constexpr int WARP_SMEM = STAGES * IN_BYTES + OUT_BUFS * OUT_BYTES;
    static constexpr int SMEM = WARPS * WARP_SMEM + WARPS * STAGES * 8 + 1024;
};

template <int SCH>
struct ReduceCfg {
    static constexpr int WARPS = 8;
    static constexpr int IN_SEG = (SCH == S_ASYM4) ? 32 : 64;
    static constexpr int OUT_SEG = 256;
    static constexpr int STAGES = (SCH == S_ASYM4) ? 12 : 8;
    static constexpr int IN_BYTES = 32 * IN_SEG;
    static constexpr int OUT_BYTES = 32 * OUT_SEG;
    static constexpr int OUT_BUFS = 1;
    static constexpr int WARP_SMEM = STAGES * IN_BYTES + OUT_BUFS * OUT_BYTES;
    static constexpr int SMEM = WARPS * WARP_SMEM + WARPS * STAGES * 8 + 1024;
};

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw)
{
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// ------------------------------------------------------------ segment I/O
// Read this lane's 64-element input segment (row `lane` of a stage).
template <int IN>
__device__ __forceinline__ void load_segment(const uint8_t* st, int lane, float (&v)[SEG])
{
    if constexpr (IN == IN_FP32) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint8_t* box = st + h * 4096;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint4 w = lds128(box, sw128(lane, c));
                v[h * 32 + c * 4 + 0] = __uint_as_float(w.x);
                v[h * 32 + c * 4 + 1] = __uint_as_float(w.y);
                v[h * 32 + c * 4 + 2] = __uint_as_float(w.z);
                v[h * 32 + c * 4 + 3] = __uint_as_float(w.w);
            }
        }
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 w = lds128(st, sw128(lane, c));
            uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if constexpr (IN == IN_BF16) {
                    v[c * 8 + 2 * k] = bf16lo(ws[k]);
                    v[c * 8 + 2 * k + 1] = bf16hi(ws[k]);
                } else {
                    float2 f = f16x2_to_f32(ws[k]);
                    v[c * 8 + 2 * k] = f.x;
                    v[c * 8 + 2 * k + 1] = f.y;
                }
            }
        }
    }
}

// Write this lane's 64-element output row into a staging buffer.
template <int OUT>
__device__ __forceinline__ void store_segment(uint8_t* ob, int lane, const float (&v)[SEG])
{
    if constexpr (OUT == IN_FP32) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int e = h * 32 + c * 4;
                sts128(ob + h * 4096, sw128(lane, c),
                       make_uint4(__float_as_uint(v[e]), __float_as_uint(v[e + 1]),
                                  __float_as_uint(v[e + 2]), __float_as_uint(v[e + 3])));
            }
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float lo = v[c * 8 + 2 * k], hi = v[c * 8 + 2 * k + 1];
                w[k] = (OUT == IN_BF16) ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
            }
            sts128(ob, sw128(lane, c), make_uint4(w[0], w[1], w[2], w[3]));
        }
    }
}

// Byte codes of one segment from a stage (64 bytes, SW64) into 16 words.
__device__ __forceinline__ void load_codes8(const uint8_t* st, int lane, uint32_t (&q)[16])
{
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 w = lds128(st, sw64(lane, c));
        q[c * 4 + 0] = w.x;
        q[c * 4 + 1] = w.y;
        q[c * 4 + 2] = w.z;
        q[c * 4 + 3] = w.w;
    }
}

// Nibble codes of one segment (32 bytes, SW32) into 8 words.
__device__ __forceinline__ void load_codes4(const uint8_t* st, int lane, uint32_t (&q)[8])
{
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint4 w = lds128(st, sw32(lane, c));
        q[c * 4 + 0] = w.x;
        q[c * 4 + 1] = w.y;
        q[c * 4 + 2] = w.z;
        q[c * 4 + 3] = w.w;
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

// Per-tensor amax accumulation for the dual-scale state: a running max per
// warp while consecutive warp tiles stay inside one tensor, flushed with one
// atomicMax (non-negative floats order like their bit patterns).
struct AmaxTracker {
    int tensor = -1;
    float m = 0.0f;

    __device__ __forceinline__ void flush(float* state, int lane)
    {
        const uint32_t w = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
        if (lane == 0 && tensor >= 0 && w != 0u)
            atomicMax(reinterpret_cast<unsigned int*>(state + 2 * tensor + 1), w);
        m = 0.0f;
    }
};

// ------------------------------------------------------------ compress
// taco_compress / qar_requant / CURRENT-mode amax pre-pass (AMAX_ONLY).
template <int IN, int SCH, bool AMAX_ONLY>
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

    const int W = gridDim.x * C::WARPS;
    const int first = blockIdx.x * C::WARPS + warp;
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    // prologue: fill the ring
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            const int wt = first + s * W;
            if (wt >= p.n_warp_tiles) break;
            issue_in16or32<IN>(&p.in_map, wb + s * C::IN_BYTES, wt * 32, &bars[s]);
        }
    }

    AmaxTracker amax;
    int cached_tensor = -1;
    float S = 1.0f, tinv = 0.0f;
    const int L = p.lanes_per_block;
    int stage = 0;
    uint32_t phase = 0;
    int k = 0;
    bool aborted = false;

    for (int wt = first; wt < p.n_warp_tiles; wt += W, ++k) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[stage], phase, p.err));
        if (!ok) {
            aborted = true;
            break;
        }
        float v[SEG];
        load_segment<IN>(wb + stage * C::IN_BYTES, lane, v);
        __syncwarp();
        // refill this stage with the tile STAGES ahead
        {
            const int nwt = wt + C::STAGES * W;
            if (nwt < p.n_warp_tiles) {
                if (lane == 0) {
                    fence_proxy_async_smem();
                    issue_in16or32<IN>(&p.in_map, wb + stage * C::IN_BYTES, nwt * 32, &bars[stage]);
                }
            }
        }
        if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
        }

        const int g = wt * 32 + lane;     // global segment of this lane
        const bool valid = g < p.M;

        uint32_t out_words[16];
        if constexpr (SCH == S_TACO) {
            // per-tensor state of this warp tile
            const int g_last = min(wt * 32 + 31, p.M - 1);
            const int t_first = (int)fdiv((uint32_t)(wt * 32), p.seg_per_tensor);
            const int t_last = (int)fdiv((uint32_t)g_last, p.seg_per_tensor);
            const bool uniform = (t_first == t_last);
            const int tens = uniform ? t_first : (int)fdiv((uint32_t)min(g, p.M - 1), p.seg_per_tensor);
            fwht64_local(v);
            fwht_cross(v, L, lane);
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < SEG; ++i) a = fmaxf(a, fabsf(v[i]));
            if (uniform) {
                if (tens != amax.tensor) {
                    amax.flush(p.state, lane);
                    amax.tensor = tens;
                }
                amax.m = fmaxf(amax.m, a);
            } else if (valid && a > 0.0f) {
                atomicMax(reinterpret_cast<unsigned int*>(p.state + 2 * tens + 1), __float_as_uint(a));
            }
            if constexpr (AMAX_ONLY) {
                continue;
            } else {
                if (!uniform || tens != cached_tensor) {
                    S = __ldg(p.state + 2 * tens);
                    tinv = __frcp_rn(__fmul_rn(448.0f, S));
                    cached_tensor = uniform ? tens : -1;
                }
                const float ab = group_max(a, L);
                uint32_t r = e4m3_encode(__fmul_rn(ab, tinv));
                if (r == 0u && ab > 0.0f) r = 1u;
                const float sb = __fmul_rn(S, e4m3_decode(r));
                const float inv = (sb > 0.0f) ? __frcp_rn(sb) : 0.0f;
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    const uint32_t lo = e4m3x2_encode(__fmul_rn(v[4 * w], inv), __fmul_rn(v[4 * w + 1], inv));
                    const uint32_t hi = e4m3x2_encode(__fmul_rn(v[4 * w + 2], inv), __fmul_rn(v[4 * w + 3], inv));
                    out_words[w] = lo | (hi << 16);
                }
                if (valid && (lane & (L - 1)) == 0)
                    static_cast<uint8_t*>(p.scales)[g >> p.lanes_log2] = static_cast<uint8_t>(r);
            }
        } else if constexpr (SCH == S_INT8SYM) {
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < SEG; ++i) a = fmaxf(a, fabsf(v[i]));
            const float s = __fdiv_rn(a, 127.0f);
            const float inv = (a > 0.0f) ? __fdiv_rn(127.0f, a) : 0.0f;
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                uint32_t word = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    int q = __float2int_rn(__fmul_rn(v[4 * w + b], inv));
                    q = max(-127, min(127, q));
                    word |= (static_cast<uint32_t>(q) & 0xffu) << (8 * b);
                }
                out_words[w] = word;
            }
            if (valid) static_cast<float*>(p.scales)[g] = s;
        } else {
            constexpr int Q = (SCH == S_ASYM4) ? 15 : 255;
            float mn = v[0], mx = v[0];
#pragma unroll
            for (int i = 1; i < SEG; ++i) {
                mn = fminf(mn, v[i]);
                mx = fmaxf(mx, v[i]);
            }
            mn = group_min(mn, 2);
            mx = group_max(mx, 2);
            float sf = __fdiv_rn(__fsub_rn(mx, mn), (float)Q);
            sf = fminf(sf, 65504.0f);
            const __half s16 = __float2half_rn(sf);
            const __half z16 = __float2half_rn(fminf(fmaxf(mn, -65504.0f), 65504.0f));
            const float s = __half2float(s16), z = __half2float(z16);
            const float inv = (s > 0.0f) ? __frcp_rn(s) : 0.0f;
            if constexpr (SCH == S_ASYM4) {
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    uint32_t word = 0;
#pragma unroll
                    for (int b = 0; b < 8; ++b) {
                        int q = __float2int_rn(__fmul_rn(__fsub_rn(v[8 * w + b], z), inv));
                        q = max(0, min(Q, q));
                        word |= static_cast<uint32_t>(q) << (4 * b);
                    }
                    out_words[w] = word;
                }
            } else {
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    uint32_t word = 0;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        int q = __float2int_rn(__fmul_rn(__fsub_rn(v[4 * w + b], z), inv));
                        q = max(0, min(Q, q));
                        word |= static_cast<uint32_t>(q) << (8 * b);
                    }
                    out_words[w] = word;
                }
            }
            if (valid && (lane & 1) == 0) {
                static_cast<__half*>(p.scales)[g >> 1] = s16;
                static_cast<__half*>(p.zeros)[g >> 1] = z16;
            }
        }

        if constexpr (!AMAX_ONLY) {
            // stage the codes and store them with one TMA per warp tile
            uint8_t* ob = outb + (k & 1) * C::OUT_BYTES;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
            if constexpr (SCH == S_ASYM4) {
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    sts128(ob, sw32(lane, c),
                           make_uint4(out_words[4 * c], out_words[4 * c + 1], out_words[4 * c + 2], out_words[4 * c + 3]));
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    sts128(ob, sw64(lane, c),
                           make_uint4(out_words[4 * c], out_words[4 * c + 1], out_words[4 * c + 2], out_words[4 * c + 3]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&p.out_map, 0, wt * 32, ob);
                bulk_commit();
            }
        }
    }
    if constexpr (SCH == S_TACO) amax.flush(p.state, lane);
    if (lane == 0) {
        bulk_wait_all();
        if (aborted) {
            // let every load this warp issued land before the CTA can exit
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < C::STAGES; ++i) {
                mbar_wait(&bars[s], ph, p.err);
                if (++s == C::STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    }
}

// ------------------------------------------------------------ decompress
template <int SCH, int OUT>
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
    const int first = blockIdx.x * C::WARPS + warp;
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
        for (int s = 0; s < C::STAGES; ++s) {
            const int wt = first + s * W;
            if (wt >= p.n_warp_tiles) break;
            mbar_arrive_expect_tx(&bars[s], C::IN_BYTES);
            tma_load_2d(wb + s * C::IN_BYTES, &p.in_map, 0, wt * 32, &bars[s]);
        }
    }
    __syncwarp();
    const int L = p.lanes_per_block;
    int stage = 0;
    uint32_t phase = 0;
    int k = 0;
    bool aborted = false;
    for (int wt = first; wt < p.n_warp_tiles; wt += W, ++k) {
        const int g = wt * 32 + lane;
        const bool valid = g < p.M;
        // metadata of this lane's segment
        float sb = 0.0f, z = 0.0f;
        if (valid) {
            if constexpr (SCH == S_TACO) {
                const int tens = (int)fdiv((uint32_t)g, p.seg_per_tensor);
                const uint32_t r = __ldg(static_cast<const uint8_t*>(p.scales) + (g >> p.lanes_log2));
                sb = __fmul_rn(__ldg(p.state + 2 * tens), e4m3_decode(r));
            } else if constexpr (SCH == S_INT8SYM) {
                sb = __ldg(static_cast<const float*>(p.scales) + g);
            } else {
                sb = __half2float(__ldg(static_cast<const __half*>(p.scales) + (g >> 1)));
                z = __half2float(__ldg(static_cast<const __half*>(p.zeros) + (g >> 1)));
            }
        }
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[stage], phase, p.err));
        if (!ok) {
            aborted = true;
            break;
        }
        float v[SEG];
        if constexpr (SCH == S_ASYM4) {
            uint32_t q[8];
            load_codes4(wb + stage * C::IN_BYTES, lane, q);
            __syncwarp();
#pragma unroll
            for (int w = 0; w < 8; ++w)
#pragma unroll
                for (int b = 0; b < 8; ++b)
                    v[8 * w + b] = __fmaf_rn(u8_to_float((q[w] >> (4 * b)) & 15u), sb, z);
        } else {
            uint32_t q[16];
            load_codes8(wb + stage * C::IN_BYTES, lane, q);
            __syncwarp();
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                if constexpr (SCH == S_TACO) {
                    const float2 lo = e4m3x2_decode(q[w] & 0xffffu);
                    const float2 hi = e4m3x2_decode(q[w] >> 16);
                    v[4 * w + 0] = __fmul_rn(lo.x, sb);
                    v[4 * w + 1] = __fmul_rn(lo.y, sb);
                    v[4 * w + 2] = __fmul_rn(hi.x, sb);
                    v[4 * w + 3] = __fmul_rn(hi.y, sb);
                } else if constexpr (SCH == S_INT8SYM) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) v[4 * w + b] = __fmul_rn(s8_to_float(q[w] >> (8 * b)), sb);
                } else {
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        v[4 * w + b] = __fmaf_rn(u8_to_float((q[w] >> (8 * b)) & 0xffu), sb, z);
                }
            }
        }
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
            fwht64_local(v);
            fwht_cross(v, L, lane);
#pragma unroll
            for (int i = 0; i < SEG; ++i) v[i] = __fmul_rn(v[i], p.inv_block);
        }
        uint8_t* ob = outb + (k & 1) * C::OUT_BYTES;
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
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
        if (aborted) {
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < C::STAGES; ++i) {
                mbar_wait(&bars[s], ph, p.err);
                if (++s == C::STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    }
}

// ------------------------------------------------------------ reduce
// Units of the stage ring are (warp tile, rank) pairs, rank fastest.
template <int SCH>
__device__ __forceinline__ void reduce_issue(const ReduceParams& p, uint8_t* wb, uint64_t* bars,
                                             int stage, int unit, int first, int W)
{
    using C = ReduceCfg<SCH>;
    const int t = unit / p.n_ranks, r = unit - t * p.n_ranks;
    const int wt = first + t * W;
    mbar_arrive_expect_tx(&bars[stage], C::IN_BYTES);
    tma_load_2d(wb + stage * C::IN_BYTES, &p.in_map[r], 0, p.seg_begin + wt * 32, &bars[stage]);
}

template <int SCH>
__global__ void __launch_bounds__(ReduceCfg<SCH>::WARPS * 32, 1)
reduce_kernel(const __grid_constant__ ReduceParams p)
{
    using C = ReduceCfg<SCH>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = aligned_smem(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* wb = smem + warp * C::WARP_SMEM;
    uint8_t* outb = wb + C::STAGES * C::IN_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::WARPS * C::WARP_SMEM) + warp * C::STAGES;
    const int W = gridDim.x * C::WARPS;
    const int first = blockIdx.x * C::WARPS + warp;
    const int n = p.n_ranks;
    const int my_tiles = (first < p.n_warp_tiles) ? (p.n_warp_tiles - first + W - 1) / W : 0;
    const int total_units = my_tiles * n;
    if (lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
        for (int u = 0; u < C::STAGES && u < total_units; ++u) reduce_issue<SCH>(p, wb, bars, u, u, first, W);
    }
    __syncwarp();
    float Sr[MAX_RANKS];
    if constexpr (SCH == S_TACO) {
#pragma unroll
        for (int r = 0; r < MAX_RANKS; ++r) Sr[r] = (r < n) ? __ldg(p.state[r]) : 0.0f;
    }
    const int L = p.lanes_per_block;
    int stage = 0;
    uint32_t phase = 0;
    int unit = 0;
    bool aborted = false;
    for (int t = 0; t < my_tiles && !aborted; ++t) {
        const int wt = first + t * W;
        const int o = wt * 32 + lane;          // output segment
        const bool valid = o < p.M_out;
        const int g = p.seg_begin + o;         // input segment
        float sc[MAX_RANKS], zz[MAX_RANKS];
#pragma unroll
        for (int r = 0; r < MAX_RANKS; ++r) {
            sc[r] = 0.0f;
            zz[r] = 0.0f;
            if (r < n && valid) {
                if constexpr (SCH == S_TACO) {
                    const uint32_t b = __ldg(static_cast<const uint8_t*>(p.scales[r]) + (g >> p.lanes_log2));
                    sc[r] = __fmul_rn(Sr[r], e4m3_decode(b));
                } else if constexpr (SCH == S_INT8SYM) {
                    sc[r] = __ldg(static_cast<const float*>(p.scales[r]) + g);
                } else {
                    sc[r] = __half2float(__ldg(static_cast<const __half*>(p.scales[r]) + (g >> 1)));
                    zz[r] = __half2float(__ldg(static_cast<const __half*>(p.zeros[r]) + (g >> 1)));
                }
            }
        }
        float acc[SEG];
#pragma unroll
        for (int r = 0; r < MAX_RANKS; ++r) {
            if (r >= n) break;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[stage], phase, p.err));
            if (!ok) {
                aborted = true;
                break;
            }
            float v[SEG];
            if constexpr (SCH == S_ASYM4) {
                uint32_t q[8];
                load_codes4(wb + stage * C::IN_BYTES, lane, q);
                __syncwarp();
#pragma unroll
                for (int w = 0; w < 8; ++w)
#pragma unroll
                    for (int b = 0; b < 8; ++b)
                        v[8 * w + b] = __fmaf_rn(u8_to_float((q[w] >> (4 * b)) & 15u), sc[r], zz[r]);
            } else {
                uint32_t q[16];
                load_codes8(wb + stage * C::IN_BYTES, lane, q);
                __syncwarp();
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    if constexpr (SCH == S_TACO) {
                        const float2 lo = e4m3x2_decode(q[w] & 0xffffu);
                        const float2 hi = e4m3x2_decode(q[w] >> 16);
                        v[4 * w + 0] = __fmul_rn(lo.x, sc[r]);
                        v[4 * w + 1] = __fmul_rn(lo.y, sc[r]);
                        v[4 * w + 2] = __fmul_rn(hi.x, sc[r]);
                        v[4 * w + 3] = __fmul_rn(hi.y, sc[r]);
                    } else if constexpr (SCH == S_INT8SYM) {
#pragma unroll
                        for (int b = 0; b < 4; ++b) v[4 * w + b] = __fmul_rn(s8_to_float(q[w] >> (8 * b)), sc[r]);
                    } else {
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            v[4 * w + b] = __fmaf_rn(u8_to_float((q[w] >> (8 * b)) & 0xffu), sc[r], zz[r]);
                    }
                }
            }
            // refill this stage
            if (lane == 0 && unit + C::STAGES < total_units) {
                fence_proxy_async_smem();
                reduce_issue<SCH>(p, wb, bars, stage, unit + C::STAGES, first, W);
            }
            ++unit;
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
            if (r == 0) {
#pragma unroll
                for (int i = 0; i < SEG; ++i) acc[i] = v[i];
            } else {
#pragma unroll
                for (int i = 0; i < SEG; ++i) acc[i] = __fadd_rn(acc[i], v[i]);
            }
        }
        if (aborted) break;
        if constexpr (SCH == S_TACO) {
            fwht64_local(acc);
            fwht_cross(acc, L, lane);
#pragma unroll
            for (int i = 0; i < SEG; ++i) acc[i] = __fmul_rn(acc[i], p.inv_block);
        }
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        store_segment<IN_FP32>(outb, lane, acc);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            store_out16or32<IN_FP32>(&p.out_map, outb, wt * 32);
            bulk_commit();
        }
    }
    if (lane == 0) {
        bulk_wait_all();
        if (aborted) {
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < C::STAGES; ++i) {
                mbar_wait(&bars[s], ph, p.err);
                if (++s == C::STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    }
}

// ------------------------------------------------------------ small kernels
enum StateOp : int { STATE_UPDATE = 0, STATE_RESET_AMAX = 1, STATE_SET_SCALE = 2 };

__global__ void state_kernel(float* state, long long n, int op);
__global__ void copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long n16);

}  // namespace qta
