// qta_device.cuh -- device building blocks of the codec kernels (sm_103a):
// mbarrier / TMA (cp.async.bulk.tensor) primitives with bounded waits, the
// swizzled shared-memory addressing that matches the TMA swizzle modes, the
// number-format conversions, and the register-resident block Hadamard.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace qta {

// ----------------------------------------------------------------------------
// Work decomposition.  A "segment" is 64 consecutive elements of the flat
// tensor: the unit one lane transforms / quantizes.  Blocks of 64/128/256
// elements span 1/2/4 segments held by adjacent lanes.
// ----------------------------------------------------------------------------
constexpr int SEG = 64;
constexpr int MAX_RANKS = 16;

enum : uint32_t { ERR_WAIT_TIMEOUT = 1u };

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most ~2 s.
// Returns false (and ORs ERR_WAIT_TIMEOUT into *err) when the limit is hit.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, unsigned int* err)
{
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > 2000000000ull) {
            atomicOr(err, ERR_WAIT_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* err)
{
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, err);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1, const void* src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(map), "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int c0, int c1, int c2,
                                             const void* src)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to TMA.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// -------------------------------------------- swizzled shared-memory rows
// TMA with SWIZZLE_{128,64,32}B stores the 16-byte chunk c of smem row t at
// chunk c ^ f(t) (bits [7,10) / [7,9) / [7,8) of the byte address XORed into
// bits [4,7) / [4,6) / [4,5)).  Each thread owns one row (its segment), so
// these layouts make its 16-byte accesses bank-conflict free.
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t c) { return row * 128u + ((c ^ (row & 7u)) << 4); }
__device__ __forceinline__ uint32_t sw64(uint32_t row, uint32_t c) { return row * 64u + ((c ^ ((row >> 1) & 3u)) << 4); }
__device__ __forceinline__ uint32_t sw32(uint32_t row, uint32_t c) { return row * 32u + ((c ^ ((row >> 2) & 1u)) << 4); }

__device__ __forceinline__ uint4 lds128(const uint8_t* base, uint32_t off)
{
    return *reinterpret_cast<const uint4*>(base + off);
}

__device__ __forceinline__ void sts128(uint8_t* base, uint32_t off, uint4 v)
{
    *reinterpret_cast<uint4*>(base + off) = v;
}

// ---------------------------------------------------------------- formats
// FP8 E4M3 pair encode, round-to-nearest-even with saturation to +-448
// (cvt .satfinite); lo goes to the low byte.
__device__ __forceinline__ uint32_t e4m3x2_encode(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t e4m3_encode(float v) { return e4m3x2_encode(v, 0.0f) & 0xffu; }

// FP8 E4M3 pair decode (exact): the low byte gives .x.
__device__ __forceinline__ float2 e4m3x2_decode(uint32_t two_codes)
{
    uint32_t h2;
    uint16_t in = static_cast<uint16_t>(two_codes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    __half2 h = *reinterpret_cast<__half2*>(&h2);
    return __half22float2(h);
}

__device__ __forceinline__ float e4m3_decode(uint32_t code) { return e4m3x2_decode(code & 0xffu).x; }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float2 f16x2_to_f32(uint32_t w)
{
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Exact small-integer to float without the conversion pipe: the bits
// 0x4B000000 | u are the float 2^23 + u for u < 2^23.
__device__ __forceinline__ float u8_to_float(uint32_t u) { return __fsub_rn(__uint_as_float(0x4B000000u | u), 8388608.0f); }
// Signed int8 held in the low byte of b (two's complement).
__device__ __forceinline__ float s8_to_float(uint32_t b) { return __fsub_rn(__uint_as_float(0x4B000000u | ((b & 0xffu) ^ 0x80u)), 8388736.0f); }

// Per-tensor scale rule: S = amax/448, or 1 when that is zero, non-finite or
// below the smallest normal float.
__device__ __forceinline__ float scale_from_amax(float amax)
{
    float S = __fdiv_rn(amax, 448.0f);
    if (!(S >= 1.17549435e-38f && S <= 3.40282347e+38f)) S = 1.0f;
    return S;
}

// ---------------------------------------------------------------- Hadamard
// Butterfly stages with strides 1..32 inside one thread's 64 values, in
// ascending order; each pair (j, j+h) -> (a+b, a-b) in binary32.
__device__ __forceinline__ void fwht64_local(float (&v)[SEG])
{
#pragma unroll
    for (int h = 1; h < SEG; h <<= 1) {
#pragma unroll
        for (int i = 0; i < SEG; i += 2 * h) {
#pragma unroll
            for (int j = i; j < i + h; ++j) {
                const float a = v[j], b = v[j + h];
                v[j] = __fadd_rn(a, b);
                v[j + h] = __fsub_rn(a, b);
            }
        }
    }
}

// Remaining stages (strides 64, 128) across the 2 or 4 lanes that hold one
// block: the lower lane of a pair keeps a+b, the upper keeps a-b, where a is
// the lower lane's value.
__device__ __forceinline__ void fwht_cross(float (&v)[SEG], int lanes_per_block, int lane)
{
    for (int d = 1; d < lanes_per_block; d <<= 1) {
        const bool upper = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < SEG; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, v[i], d);
            v[i] = upper ? __fsub_rn(o, v[i]) : __fadd_rn(v[i], o);
        }
    }
}

__device__ __forceinline__ float group_max(float m, int lanes_per_block)
{
    for (int d = 1; d < lanes_per_block; d <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    return m;
}

__device__ __forceinline__ float group_min(float m, int lanes_per_block)
{
    for (int d = 1; d < lanes_per_block; d <<= 1) m = fminf(m, __shfl_xor_sync(0xffffffffu, m, d));
    return m;
}

}  // namespace qta
