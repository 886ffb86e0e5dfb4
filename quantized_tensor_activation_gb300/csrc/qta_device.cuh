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

// Wait for the phase with the given parity to complete until the
// %globaltimer value `deadline_ns`; false when the deadline passes first.
static __device__ __noinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, uint64_t deadline_ns)
{
    for (;;) {
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() > deadline_ns) return false;
    }
}

// ------------------------------------------- programmatic dependent launch
// The kernels are launched with programmatic stream serialization: a kernel
// may start while its predecessor on the stream drains.  Every thread waits
// for the predecessor's completion (and memory) before its first global
// access; the trigger lets the successor be scheduled as SMs free up.  Both
// are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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

// ---------------------------------------------------------------- packed FP32
// Values travel as pairs of binary32 in one 64-bit register: pair j of a
// segment holds elements (2j, 2j+1).  add/sub/mul/fma .f32x2 round each lane
// to nearest-even exactly like the scalar instructions, at one instruction
// per pair.
using u64 = unsigned long long;

__device__ __forceinline__ u64 pk2(float lo, float hi)
{
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 up2(u64 v)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

__device__ __forceinline__ u64 add2(u64 a, u64 b)
{
    u64 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ u64 sub2(u64 a, u64 b)
{
    u64 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ u64 mul2(u64 a, u64 b)
{
    u64 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c)
{
    u64 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float min3f(float a, float b, float c)
{
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ---------------------------------------------------------------- formats
// FP8 E4M3 pair encode, round-to-nearest-even with saturation to +-448
// (cvt .satfinite); lo goes to the low byte.
__device__ __forceinline__ uint16_t e4m3x2_encode(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t e4m3_encode(float v) { return e4m3x2_encode(v, 0.0f) & 0xffu; }

__device__ __forceinline__ uint32_t join16(uint16_t lo, uint16_t hi)
{
    uint32_t r;
    asm("mov.b32 %0, {%1, %2};" : "=r"(r) : "h"(lo), "h"(hi));
    return r;
}

// FP8 E4M3 pair decode (exact) to a float pair: the low byte gives .x.
__device__ __forceinline__ u64 e4m3x2_decode(uint16_t two_codes)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two_codes));
    const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h2));
    return pk2(f.x, f.y);
}

__device__ __forceinline__ float e4m3_decode(uint32_t code)
{
    return up2(e4m3x2_decode(static_cast<uint16_t>(code & 0xffu))).x;
}

__device__ __forceinline__ uint16_t lo16(uint32_t w) { return static_cast<uint16_t>(w & 0xffffu); }
__device__ __forceinline__ uint16_t hi16(uint32_t w) { return static_cast<uint16_t>(w >> 16); }

__device__ __forceinline__ u64 bf16x2_to_pair(uint32_t w) { return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)); }

__device__ __forceinline__ u64 f16x2_to_pair(uint32_t w)
{
    const float2 f = __half22float2(*reinterpret_cast<__half2*>(&w));
    return pk2(f.x, f.y);
}

__device__ __forceinline__ uint32_t pair_to_bf16x2(u64 v)
{
    const float2 f = up2(v);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y), "f"(f.x));
    return r;
}

__device__ __forceinline__ uint32_t pair_to_f16x2(u64 v)
{
    const float2 f = up2(v);
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y), "f"(f.x));
    return r;
}

// Small integers to float without the conversion pipe: the bits
// 0x4B000000 | u are the float 2^23 + u for u < 2^23.  Byte k of `w` (k = 0..3)
// goes to the low byte via PRMT.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Four unsigned bytes of w as two float pairs (exact): (b0, b1), (b2, b3).
__device__ __forceinline__ void u8x4_to_pairs(uint32_t w, u64& p01, u64& p23)
{
    const uint32_t magic = 0x4B000000u;
    const u64 off = pk2(8388608.0f, 8388608.0f);
    // prmt selectors: byte 0..3 of w into the low byte, bytes 1..3 from magic (b = magic: bytes 4..7)
    p01 = sub2(pk2(__uint_as_float(prmt(w, magic, 0x7650u)), __uint_as_float(prmt(w, magic, 0x7651u))), off);
    p23 = sub2(pk2(__uint_as_float(prmt(w, magic, 0x7652u)), __uint_as_float(prmt(w, magic, 0x7653u))), off);
}

// Four signed (two's complement) bytes of w as two float pairs (exact).
__device__ __forceinline__ void s8x4_to_pairs(uint32_t w, u64& p01, u64& p23)
{
    const u64 off = pk2(8388736.0f, 8388736.0f);  // 2^23 + 128
    const uint32_t wb = w ^ 0x80808080u;           // b + 128 for each signed byte
    const uint32_t magic = 0x4B000000u;
    p01 = sub2(pk2(__uint_as_float(prmt(wb, magic, 0x7650u)), __uint_as_float(prmt(wb, magic, 0x7651u))), off);
    p23 = sub2(pk2(__uint_as_float(prmt(wb, magic, 0x7652u)), __uint_as_float(prmt(wb, magic, 0x7653u))), off);
}

// Eight nibbles of w (element i in bits 4i..4i+3) dequantized as
// f[i] = fmaf(n_i, s, z) with s an fp16 scale and z a widened fp16 zero.
// A nibble n OR'd under the fp16 pattern 0x6400 is 1024 + n (or 1024 + 16n
// for an upper nibble of a byte), so one LOP3 yields two fp16 values and
// one f16x2 subtract (or fma by 1/16, -64) leaves n exactly.  The
// mixed-precision fma.rn.f32.f16 multiplies two fp16 operands exactly and
// adds the f32 zero with one rounding: fmaf(n, s, z) bit for bit.
__device__ __forceinline__ void fma_f16_pair(uint32_t q2, uint16_t s, float z, float& lo, float& hi)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "fma.rn.f32.f16 %0, l, %3, %4;\n\tfma.rn.f32.f16 %1, h, %3, %4;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(q2), "h"(s), "f"(z));
}

__device__ __forceinline__ void u4x8_dequant(uint32_t w, uint16_t s, float z, float (&f)[8])
{
    const uint32_t w8 = w >> 8;
    uint32_t h04 = (w & 0x000F000Fu) | 0x64006400u;    // 1024 + n0, 1024 + n4
    uint32_t h15 = (w & 0x00F000F0u) | 0x64006400u;    // 1024 + 16 n1, 1024 + 16 n5
    uint32_t h26 = (w8 & 0x000F000Fu) | 0x64006400u;   // 1024 + n2, 1024 + n6
    uint32_t h37 = (w8 & 0x00F000F0u) | 0x64006400u;   // 1024 + 16 n3, 1024 + 16 n7
    const uint32_t k1024 = 0x64006400u, k16th = 0x2C002C00u, km64 = 0xD400D400u;
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(h04) : "r"(k1024));
    asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(h26) : "r"(k1024));
    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(h15) : "r"(k16th), "r"(km64));
    asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(h37) : "r"(k16th), "r"(km64));
    fma_f16_pair(h04, s, z, f[0], f[4]);
    fma_f16_pair(h15, s, z, f[1], f[5]);
    fma_f16_pair(h26, s, z, f[2], f[6]);
    fma_f16_pair(h37, s, z, f[3], f[7]);
}

// The same values scaled by 2^-24 (the low nibble of each byte) and 2^-20
// (the high nibble), for a sum that is scaled back once at its end.  A
// nibble masked in place, without the magic pattern, is the fp16 subnormal
// n 2^-24 (low) or 16 n 2^-24 = n 2^-20 (high): one AND yields two fp16
// operands and nothing is subtracted.  With zlo = z 2^-24 and zhi = z 2^-20
// (exact), the mixed-precision fma gives RN(2^-24 (n s + z)).  s and z are
// fp16 values, so n s + z is a multiple of 2^-24 and its scaled value is zero
// or a normal FP32 number: the rounding commutes with the power-of-two scale,
// and the result is 2^-24 fmaf(n, s, z) bit for bit.
__device__ __forceinline__ void u4x8_dequant_scaled(uint32_t w, uint16_t s, float zlo, float zhi, float (&f)[8])
{
    const uint32_t w8 = w >> 8;
    fma_f16_pair(w & 0x000F000Fu, s, zlo, f[0], f[4]);    // n0, n4 (2^-24)
    fma_f16_pair(w & 0x00F000F0u, s, zhi, f[1], f[5]);    // n1, n5 (2^-20)
    fma_f16_pair(w8 & 0x000F000Fu, s, zlo, f[2], f[6]);   // n2, n6
    fma_f16_pair(w8 & 0x00F000F0u, s, zhi, f[3], f[7]);   // n3, n7
}

// Round-to-nearest-even to an integer through the FP32 adder: for |y| < 2^22
// the bits of y + 1.5*2^23 are 0x4B400000 + rint(y); the low byte of those
// bits is rint(y) mod 256.
__device__ __forceinline__ u64 rint_bits2(u64 y)
{
    return add2(y, pk2(12582912.0f, 12582912.0f));
}

// Round to the nearest integer (ties to even), saturating at the int32 range;
// NaN gives 0.
__device__ __forceinline__ uint32_t cvt_rni_s32(float y)
{
    uint32_t r;
    asm("cvt.rni.s32.f32 %0, %1;" : "=r"(r) : "f"(y));
    return r;
}

// Four int32, each clamped to [0, 255], as the bytes [a b c d] of one word
// (a lowest): two saturating pack conversions.  The clamp after the rounding
// gives the codes of a rounding conversion that saturates to u8 directly.
__device__ __forceinline__ uint32_t pack4_sat_u8(uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    uint32_t hi, r;
    asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(d), "r"(c), "r"(0u));
    asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(b), "r"(a), "r"(hi));
    return r;
}

// Low bytes of four words into one word: (a, b, c, d) -> bytes [a b c d].
__device__ __forceinline__ uint32_t bytes4(uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    return prmt(prmt(a, b, 0x7740u), prmt(c, d, 0x7740u), 0x5410u);
}

__device__ __forceinline__ uint32_t lo32(u64 v) { return static_cast<uint32_t>(v); }
__device__ __forceinline__ uint32_t hi32(u64 v) { return static_cast<uint32_t>(v >> 32); }

// Per-tensor scale rule: S = amax/448, or 1 when that is zero, non-finite or
// below the smallest normal float.
__device__ __forceinline__ float scale_from_amax(float amax)
{
    float S = __fdiv_rn(amax, 448.0f);
    if (!(S >= 1.17549435e-38f && S <= 3.40282347e+38f)) S = 1.0f;
    return S;
}

// ---------------------------------------------------------------- Hadamard
// Butterfly stages with strides 1, 2, 4, ..., 32 inside one lane's 64 values
// (32 pairs), ascending; each (j, j+h) -> (a+b, a-b) in binary32.  Stride 1
// pairs the two halves of a register pair (scalar); strides 2..32 pair whole
// register pairs (packed).
__device__ __forceinline__ void fwht64_local(u64 (&v)[32])
{
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float2 t = up2(v[j]);
        v[j] = pk2(__fadd_rn(t.x, t.y), __fsub_rn(t.x, t.y));
    }
#pragma unroll
    for (int hp = 1; hp < 32; hp <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 2 * hp) {
#pragma unroll
            for (int j = i; j < i + hp; ++j) {
                const u64 a = v[j], b = v[j + hp];
                v[j] = add2(a, b);
                v[j + hp] = sub2(a, b);
            }
        }
    }
}

// Remaining stages (strides 64, 128) across the 2 or 4 lanes that hold one
// block.  With a = the lower lane's value and b = the upper lane's, the lower
// lane keeps fma(a, +1, b) = a+b and the upper fma(b, -1, a) = a-b: one
// rounding each, identical to the add / subtract.
__device__ __forceinline__ void fwht_cross(u64 (&v)[32], int lanes_per_block, int lane)
{
    for (int d = 1; d < lanes_per_block; d <<= 1) {
        const float sgn = (lane & d) ? -1.0f : 1.0f;
        const u64 s2 = pk2(sgn, sgn);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const u64 o = __shfl_xor_sync(0xffffffffu, v[j], d);
            v[j] = fma2(v[j], s2, o);
        }
    }
}

// Halved exchange ("exchange layout").  In the cross-lane stages above every
// lane ships all 64 of its values to its partner.  Here each lane ships only
// the half whose outputs it does not keep, so a stage costs 32 shuffles
// instead of 64, and afterwards the lanes of a block own a block-wide strip
// of positions in every row rather than a row each.  To let both partners ship
// the same registers, lane c of a block keeps position j of its row in slot
// j ^ xm(c), c the lane's position in its block: xm = 32 c with 2 lanes per
// block.  With 4 there are two layouts.  N4 (the kernels compiled for 4-lane
// blocks): xm = 16 c, lane bit 0 mapped to xm bit 16 and lane bit 1 to xm bit
// 32, so the 8 lanes of one shared-memory wavefront read 8 different 16-byte
// bank groups of their rows under the 64- and 128-byte swizzles (the code and
// bf16 segment loads).  Otherwise (the kernels that read the block size at run
// time): xm = 32 (c & 1) + 16 (c >> 1 & 1), which gives them shorter code.
template <bool N4 = false>
__device__ __forceinline__ uint32_t xl_mask(int lanes_per_block, int lane)
{
    if constexpr (N4)
        return lanes_per_block == 4 ? (lane & 3) * 16u : (lanes_per_block == 2 ? (lane & 1) * 32u : 0u);
    return (lanes_per_block >= 2 ? (lane & 1) * 32u : 0u) | (lanes_per_block == 4 ? ((lane >> 1) & 1) * 16u : 0u);
}

// fwht64_local on the permuted slots: stages with stride 16 and 32 see the
// lower and upper position of a pair swapped in the lanes whose mask has that
// bit.  With A, B the slots of a pair and s = -1 in those lanes (else +1):
// A' = fma(A, s, B), B' = fma(B, -s, A), which is (a+b, a-b) in position
// order with one rounding each, identical to the add / subtract.
__device__ __forceinline__ void fwht64_local_xl(u64 (&v)[32], uint32_t xm)
{
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float2 t = up2(v[j]);
        v[j] = pk2(__fadd_rn(t.x, t.y), __fsub_rn(t.x, t.y));
    }
#pragma unroll
    for (int hp = 1; hp < 8; hp <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 2 * hp) {
#pragma unroll
            for (int j = i; j < i + hp; ++j) {
                const u64 a = v[j], b = v[j + hp];
                v[j] = add2(a, b);
                v[j + hp] = sub2(a, b);
            }
        }
    }
#pragma unroll
    for (int hp = 8; hp < 32; hp <<= 1) {
        const float s = (xm & (2u * hp)) ? -1.0f : 1.0f;
        const u64 s2 = pk2(s, s), ns2 = pk2(-s, -s);
#pragma unroll
        for (int i = 0; i < 32; i += 2 * hp) {
#pragma unroll
            for (int j = i; j < i + hp; ++j) {
                const u64 a = v[j], b = v[j + hp];
                v[j] = fma2(a, s2, b);
                v[j + hp] = fma2(b, ns2, a);
            }
        }
    }
}

// One cross-lane stage of the halved exchange, on the permuted slots: lane c
// pairs with c ^ d.  Registers come in groups of 2H; each lane keeps the lower
// H registers of every group and ships the upper H, which hold the partner's
// kept positions (the xm bit of lane bit d sets which half that is).  With
// a = the lane's kept value and o = the partner's value at the same
// position, the pair's outputs are (lower + upper, lower - upper), each
// rounded once as in fwht_cross.
// SWAP = false: every lane writes the sum to the kept register and the
// difference to the shipped one: a + o, and fma(o, s, -s*a) with s = +1 in
// the lane that holds the upper row (else -1), which is lower - upper in both
// lanes (-s*a is exact).
// SWAP = true: the lane whose stage bit is clear (a from the lower row)
// writes fma(a, +1, o) and fma(o, -1, a); the lane whose bit is set (a from
// the upper row) writes the difference first, fma(a, -1, o) = o - a, then
// fma(o, +1, a) = o + a.  The same adds and subtracts, zero signs included,
// one instruction fewer per register pair, and the rows of the pair swapped
// in the lanes whose stage bit is set.
template <bool SWAP, int H>
__device__ __forceinline__ void xl_stage(u64 (&v)[32], int lane, int d)
{
    if constexpr (SWAP) {
        const float s = (lane & d) ? -1.0f : 1.0f;
        const u64 s2 = pk2(s, s), ns2 = pk2(-s, -s);
#pragma unroll
        for (int h = 0; h < 32; h += 2 * H)
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const u64 o = __shfl_xor_sync(0xffffffffu, v[h + H + j], d);
                const u64 a = v[h + j];
                v[h + j] = fma2(a, s2, o);
                v[h + H + j] = fma2(o, ns2, a);
            }
    } else {
        const float s = (lane & d) ? 1.0f : -1.0f;
        const u64 s2 = pk2(s, s), ns2 = pk2(-s, -s);
#pragma unroll
        for (int h = 0; h < 32; h += 2 * H)
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const u64 o = __shfl_xor_sync(0xffffffffu, v[h + H + j], d);
                const u64 a = v[h + j];
                v[h + j] = add2(a, o);
                v[h + H + j] = fma2(o, s2, mul2(a, ns2));
            }
    }
}

// Strides 64 and 128 with the halved exchange.  With 2 lanes per block, the
// stride-64 stage pairs lane c with c ^ 1 and ships registers 16-31 (xm bit
// 32).  With 4 and N4 (xm = 16 c), the stride-64 stage (c ^ 1) ships
// registers 8-15 and 24-31 (xm bit 16), then the stride-128 stage (c ^ 2)
// ships registers 16-31 (xm bit 32).  Without N4 the stride-64 stage ships
// registers 16-31 and the stride-128 stage 8-15 and 24-31.  Afterwards lane c
// of a block holds positions xm .. xm + 64/L - 1 of every row of the block in
// register groups of 32 / L registers (xl_group_row gives the row of each).
// Register 2i+t of a group holds position xm + 2i + t.
template <bool SWAP = false, bool N4 = false>
__device__ __forceinline__ void fwht_cross_xl(u64 (&v)[32], int lanes_per_block, int lane)
{
    if constexpr (N4) {
        if (lanes_per_block == 4) xl_stage<SWAP, 8>(v, lane, 1);
        if (lanes_per_block >= 2) xl_stage<SWAP, 16>(v, lane, lanes_per_block == 4 ? 2 : 1);
    } else {
        if (lanes_per_block >= 2) xl_stage<SWAP, 16>(v, lane, 1);
        if (lanes_per_block == 4) xl_stage<SWAP, 8>(v, lane, 2);
    }
}

// Block row (0 .. lanes-1) held by register group g after fwht_cross_xl: p is
// the lane's position in its block with SWAP, 0 without.  Group g holds row g
// (N4 or 2 lanes); without N4, the 4-lane groups hold rows 0, 2, 1, 3.
template <bool N4 = false>
__device__ __forceinline__ int xl_group_row(int g, int lanes_log2, int p)
{
    if constexpr (N4) return g ^ p;
    return (lanes_log2 == 2 ? (((g & 1) << 1) | (g >> 1)) : g) ^ p;
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

// max |v| over the 64 values of a lane (NaNs ignored, 0 if none is a
// number).  The maximum is exact in any order, so it runs as four
// independent chains of eight, then two combining steps: 34 three-input max
// instead of 32, with a dependent depth of 10 instead of 32.
__device__ __forceinline__ float absmax64(const u64 (&v)[32])
{
    float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float2 t = up2(v[j]);
        m[j & 3] = max3f(m[j & 3], fabsf(t.x), fabsf(t.y));
    }
    return fmaxf(max3f(m[0], m[1], m[2]), m[3]);
}

// min and max over the 64 values of a lane (NaNs ignored), as four
// independent chains each, like absmax64.
__device__ __forceinline__ void minmax64(const u64 (&v)[32], float& mn, float& mx)
{
    float lo[4], hi[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float2 t = up2(v[c]);
        lo[c] = fminf(t.x, t.y);
        hi[c] = fmaxf(t.x, t.y);
    }
#pragma unroll
    for (int j = 4; j < 32; ++j) {
        const float2 t = up2(v[j]);
        lo[j & 3] = min3f(lo[j & 3], t.x, t.y);
        hi[j & 3] = max3f(hi[j & 3], t.x, t.y);
    }
    mn = fminf(min3f(lo[0], lo[1], lo[2]), lo[3]);
    mx = fmaxf(max3f(hi[0], hi[1], hi[2]), hi[3]);
}

}  // namespace qta
