// qta_api.cu -- the C ABI (include/qta.h): argument checks, TMA tensor maps,
// grid sizing and launches; plus the per-tensor state kernel, the copy
// kernel and the device error flags.
#include <atomic>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/qta.h"
#include "qta_launch.h"

namespace qta {

// Flags recorded by kernels whose bounded waits gave up.
__device__ unsigned int g_error_flags;

namespace {

constexpr int MAX_DEVICES = 64;

struct DeviceInfo {
    std::atomic<int> sms{0};
    std::atomic<int> smem_per_sm{0};
    std::atomic<int> smem_optin{0};
    std::atomic<unsigned int*> err{nullptr};
};
DeviceInfo g_dev[MAX_DEVICES];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t device_info(int* sms, int* smem_per_sm, unsigned int** err)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    DeviceInfo& d = g_dev[dev];
    if (d.sms.load() == 0) {
        int a = 0, b = 0, o = 0;
        if ((e = cudaDeviceGetAttribute(&a, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&b, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&o, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return e;
        d.smem_optin.store(o);
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_error_flags)) != cudaSuccess) return e;
        d.smem_per_sm.store(b);
        d.err.store(static_cast<unsigned int*>(p));
        d.sms.store(a);
    }
    *sms = d.sms.load();
    *smem_per_sm = d.smem_per_sm.load();
    *err = d.err.load();
    return cudaSuccess;
}

// Dynamic shared memory a launch may use: the opt-in maximum less a margin
// for the kernels' static shared memory (at most 64 bytes).
int smem_optin()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return 0;
    return g_dev[dev].smem_optin.load() - 256;
}

bool encoder_ready()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// 2D map over rows of `inner` elements (row stride = inner * elem bytes),
// box = {inner, box_rows rows}.
bool map_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
            uint64_t rows, CUtensorMapSwizzle sw, uint32_t box_rows = 32)
{
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * elem_bytes};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(inner), box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Segments of fp32 (256 B) as two 128-B halves: dims {32, 2, M}, box {32,1,32}.
bool map_f32(CUtensorMap* m, const void* base, uint64_t segs)
{
    cuuint64_t dims[3] = {32, 2, segs};
    cuuint64_t strides[2] = {128, 256};
    cuuint32_t box[3] = {32, 1, 32};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map of a segment array of the given dtype (input of compress, output of
// decompress).
bool map_values(CUtensorMap* m, int dtype, const void* base, uint64_t segs)
{
    if (dtype == QTA_FP32) return map_f32(m, base, segs);
    return map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, 64, segs, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Map of the codes of a segment array (8-bit: 64 B per segment; 4-bit: 32 B).
bool map_codes(CUtensorMap* m, int scheme, const void* base, uint64_t segs)
{
    if (scheme == QTA_INT4_ASYM_G128)
        return map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, 32, segs, CU_TENSOR_MAP_SWIZZLE_32B);
    return map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, 64, segs, CU_TENSOR_MAP_SWIZZLE_64B);
}

// The same 4-bit codes as rows of two segments (64 B), box = one warp tile
// (16 rows, 1 KB), 64-byte swizzle: the map of the INT4 reduce's shards.
// segs is even (a row holds a multiple of 128 codes).
bool map_codes4_rows64(CUtensorMap* m, const void* base, uint64_t segs)
{
    return map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, 64, segs / 2, CU_TENSOR_MAP_SWIZZLE_64B, 16);
}

// 1D map of n fp16 values (INT4 scales or zeros), box = 16 values (32 B).
FastDiv make_fastdiv(uint32_t d)
{
    FastDiv f;
    f.d = d;
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    f.l = l;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    return f;
}

int log2i(int v)
{
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Whether the byte ranges [a, a + na) and [b, b + nb) share a byte.
bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

size_t dtype_bytes(int32_t dt) { return dt == QTA_FP32 ? 4 : 2; }

// Scheme checks shared by every call: scheme / block combination and shape.
qta_status check_desc(const qta_desc* d)
{
    if (!d) return QTA_ERR_INVALID_ARG;
    switch (d->scheme) {
    case QTA_TACO_FP8:
        if (d->block != 64 && d->block != 128 && d->block != 256) return QTA_ERR_UNSUPPORTED;
        break;
    case QTA_INT8_SYM_B64:
        if (d->block != 64) return QTA_ERR_UNSUPPORTED;
        break;
    case QTA_INT4_ASYM_G128:
    case QTA_INT8_ASYM_G128:
        if (d->block != 128) return QTA_ERR_UNSUPPORTED;
        break;
    default: return QTA_ERR_UNSUPPORTED;
    }
    if (d->batch < 0 || d->rows < 0 || d->cols < 0 || d->max_sms < 0) return QTA_ERR_INVALID_ARG;
    if (d->cols % d->block) return QTA_ERR_INVALID_ARG;
    // element count must leave fewer than 2^31 segments
    const long double n = (long double)d->batch * (long double)d->rows * (long double)d->cols;
    if (n / 64.0L >= 2147483648.0L) return QTA_ERR_UNSUPPORTED;
    return QTA_OK;
}

int64_t n_elems(const qta_desc* d) { return d->batch * d->rows * d->cols; }

int lanes_of(const qta_desc* d)
{
    if (d->scheme == QTA_TACO_FP8) return d->block / 64;
    if (d->scheme == QTA_INT8_SYM_B64) return 1;
    return 2;
}

// Checks of one quantized tensor's buffers for a descriptor.
qta_status check_qtensor(const qta_desc* d, const qta_qtensor* q)
{
    if (!q || !q->codes || !q->scales) return QTA_ERR_INVALID_ARG;
    if (!aligned(q->codes, 16)) return QTA_ERR_ALIGNMENT;
    if (d->scheme == QTA_INT8_SYM_B64 && !aligned(q->scales, 4)) return QTA_ERR_ALIGNMENT;
    if (d->scheme == QTA_INT4_ASYM_G128 || d->scheme == QTA_INT8_ASYM_G128) {
        if (!q->zeros) return QTA_ERR_INVALID_ARG;
        if (!aligned(q->scales, 2) || !aligned(q->zeros, 2)) return QTA_ERR_ALIGNMENT;
    }
    if (d->scheme == QTA_TACO_FP8) {
        if (!q->state) return QTA_ERR_INVALID_ARG;
        if (!aligned(q->state, 4)) return QTA_ERR_ALIGNMENT;
    }
    if (q->chan) {   // the adaptive rescaling goes with the Hadamard scheme only
        if (d->scheme != QTA_TACO_FP8) return QTA_ERR_UNSUPPORTED;
        if (!aligned(q->chan, 16)) return QTA_ERR_ALIGNMENT;
    }
    return QTA_OK;
}

// Persistent grid: one CTA per SM it may use (max_sms > 0 caps the SMs, see
// qta_desc), never more CTAs than warp tiles need.  The launchers raise it to
// as many CTAs per SM as the launched kernel's registers and shared memory
// allow (persistent_grid).
int grid_for(int n_warp_tiles, int warps, int sms, int max_sms)
{
    if (max_sms > 0 && max_sms < sms) sms = max_sms;
    const int ctas = (n_warp_tiles + warps - 1) / warps;
    return ctas < sms ? ctas : sms;
}

qta_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QTA_OK : QTA_ERR_CUDA; }

}  // namespace

// The dynamic shared-memory limit of a kernel is raised once per device to
// the device's opt-in maximum less the kernel's static shared memory, so that
// launches of any size up to it (the kernel's own layout plus an optional
// copy of the channel factors) pass.
// grid_1 is one CTA per SM (grid_for).  When it spans every SM of the device
// (no max_sms cap, enough tiles) and `per_sm` CTAs of the kernel fit on an SM
// (its registers and `smem` bytes of dynamic shared memory, queried once per
// kernel), the grid grows to that many per SM, never past the CTAs the warp
// tiles need.  A capped call keeps one CTA per SM, so that its CTAs cannot
// spread over more SMs than it may use.  With the present kernels every one
// fits a single CTA per SM; the 8-warp INT8 ring hops come closest (two need
// 256 bytes more shared memory than an SM has).
int persistent_grid(const void* func, int threads, int smem, int grid_1, int n_warp_tiles, int warps,
                    std::atomic<int>* per_sm_cache)
{
    int sms = 0, smem_sm = 0;
    unsigned int* err = nullptr;
    if (device_info(&sms, &smem_sm, &err) != cudaSuccess || grid_1 < sms) return grid_1;
    int per_sm = per_sm_cache->load();
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, threads, smem) != cudaSuccess)
            per_sm = 1;
        if (per_sm < 1) per_sm = 1;
        per_sm_cache->store(per_sm);
    }
    const long long need = (static_cast<long long>(n_warp_tiles) + warps - 1) / warps;
    const long long cap = static_cast<long long>(grid_1) * per_sm;
    const long long g = need < cap ? need : cap;
    return g > grid_1 ? static_cast<int>(g) : grid_1;
}

cudaError_t ensure_smem_attr(const void* func, int smem, std::atomic<unsigned>* done_mask)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned bit = dev < 32 ? (1u << dev) : 0u;
    if (bit && (done_mask->load() & bit)) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, func);
    if (e != cudaSuccess) return e;
    const int dyn = optin - static_cast<int>(fa.sharedSizeBytes);
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn > smem ? dyn : smem);
    if (e == cudaSuccess && bit) done_mask->fetch_or(bit);
    return e;
}

__global__ void state_kernel(float* state, long long n, int op)
{
    pdl_wait();
    pdl_trigger();
    const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (t >= n) return;
    if (op == STATE_UPDATE) {
        state[2 * t] = scale_from_amax(state[2 * t + 1]);
        state[2 * t + 1] = 0.0f;
    } else if (op == STATE_RESET_AMAX) {
        state[2 * t + 1] = 0.0f;
    } else {
        state[2 * t] = scale_from_amax(state[2 * t + 1]);
    }
}

// Grid-stride 16-byte copy; each thread keeps four loads in flight.
__global__ void __launch_bounds__(512) copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                   long long n16)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
        const uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
        __stcs(dst + i, a);
        __stcs(dst + i + stride, b);
        __stcs(dst + i + 2 * stride, c);
        __stcs(dst + i + 3 * stride, d);
    }
    for (; i < n16; i += stride) __stcs(dst + i, __ldcs(src + i));
}

// Per-channel amax of the adaptive rescaling: thread t of grid column block
// owns one 16-byte vector of columns (8 16-bit or 4 fp32 values) and walks
// the rows of its row chunk, then max-accumulates into amax[] (non-negative
// floats order like their bit patterns, so max is an unsigned atomicMax).
template <int KIND>
__global__ void __launch_bounds__(256) channel_amax_kernel(const uint8_t* __restrict__ x, long long n_rows,
                                                           long long cols, long long rows_per_chunk,
                                                           float* __restrict__ amax)
{
    pdl_wait();
    pdl_trigger();
    constexpr int PER = (KIND == IN_FP32) ? 4 : 8;
    constexpr int ES = (KIND == IN_FP32) ? 4 : 2;
    const long long cv = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (cv * PER >= cols) return;
    const long long r0 = blockIdx.y * rows_per_chunk;
    const long long r1 = (r0 + rows_per_chunk < n_rows) ? r0 + rows_per_chunk : n_rows;
    float m[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) m[i] = 0.0f;
    for (long long r = r0; r < r1; ++r) {
        const uint4 w = __ldcs(reinterpret_cast<const uint4*>(x + (r * cols + cv * PER) * ES));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if constexpr (KIND == IN_FP32) {
                m[k] = fmaxf(m[k], fabsf(__uint_as_float(ws[k])));
            } else {
                const float2 f = up2((KIND == IN_BF16) ? bf16x2_to_pair(ws[k]) : f16x2_to_pair(ws[k]));
                m[2 * k] = fmaxf(m[2 * k], fabsf(f.x));
                m[2 * k + 1] = fmaxf(m[2 * k + 1], fabsf(f.y));
            }
        }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i)
        if (m[i] > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(amax + cv * PER + i), __float_as_uint(m[i]));
}

// Update of the adaptive rescaling (one CTA): E(v) = exponent field of v
// minus 127 (-127 for subnormals); E_ref = the lower median of E over the
// channels with amax > 0, found from a histogram of the 255 exponent values;
// e = min(3, max(0, E - E_ref - 2)); down = 2^-e, up = 2^e, amax = 0.
__global__ void __launch_bounds__(1024) ash_update_kernel(float* __restrict__ chan, long long cols)
{
    pdl_wait();
    pdl_trigger();
    __shared__ unsigned int hist[256];
    __shared__ int e_ref;
    float* amax = chan + 2 * cols;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
    __syncthreads();
    for (long long c = threadIdx.x; c < cols; c += blockDim.x) {
        const float v = amax[c];
        if (v > 0.0f) atomicAdd(&hist[__float_as_uint(v) >> 23], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int n = 0;
        for (int i = 0; i < 256; ++i) n += hist[i];
        int ref = 0;
        if (n > 0) {
            const unsigned int k = (n - 1) / 2;   // index of the lower median in sorted order
            unsigned int cum = 0;
            for (int i = 0; i < 256; ++i) {
                cum += hist[i];
                if (cum > k) {
                    ref = i - 127;
                    break;
                }
            }
        }
        e_ref = ref;
    }
    __syncthreads();
    const int ref = e_ref;
    for (long long c = threadIdx.x; c < cols; c += blockDim.x) {
        const float v = amax[c];
        int e = 0;
        if (v > 0.0f) {
            e = static_cast<int>(__float_as_uint(v) >> 23) - 127 - ref - 2;
            e = e < 0 ? 0 : (e > 3 ? 3 : e);
        }
        chan[c] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
        chan[cols + c] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
        amax[c] = 0.0f;
    }
}

cudaError_t launch_channel_amax(const void* x, int kind, long long n_rows, long long cols, float* amax,
                                cudaStream_t stream)
{
    const int per = kind == IN_FP32 ? 4 : 8;
    const long long ncv = cols / per;
    long long rpc = (n_rows + 65534) / 65535;   // grid.y stays within its limit
    if (rpc < 64) rpc = 64;
    const dim3 grid(static_cast<unsigned>((ncv + 255) / 256), static_cast<unsigned>((n_rows + rpc - 1) / rpc));
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    switch (kind) {
    case IN_BF16: return launch_pdl(channel_amax_kernel<IN_BF16>, grid, dim3(256), 0, stream, xb, n_rows, cols, rpc, amax);
    case IN_FP16: return launch_pdl(channel_amax_kernel<IN_FP16>, grid, dim3(256), 0, stream, xb, n_rows, cols, rpc, amax);
    case IN_FP32: return launch_pdl(channel_amax_kernel<IN_FP32>, grid, dim3(256), 0, stream, xb, n_rows, cols, rpc, amax);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_ash_update(float* chan, long long cols, cudaStream_t stream)
{
    return launch_pdl(ash_update_kernel, dim3(1), dim3(1024), 0, stream, chan, cols);
}

// Self-test of the bounded pipeline wait: one warp waits on an mbarrier
// through mbar_wait, the wait every kernel uses.  With `complete` set, one
// thread arrives first and the wait succeeds at once; otherwise nothing ever
// arrives, the wait gives up after its limit, records ERR_WAIT_TIMEOUT and
// the kernel returns normally.
__global__ void __launch_bounds__(32) wait_self_test_kernel(int complete, unsigned int* err)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (complete && threadIdx.x == 0) mbar_arrive(&bar);
    __syncwarp();
    mbar_wait(&bar, 0u, err);
}

cudaError_t launch_state(float* state, long long n, int op, cudaStream_t stream)
{
    if (n <= 0) return cudaSuccess;
    const int threads = 128;
    const long long blocks = (n + threads - 1) / threads;
    return launch_pdl(state_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, state, n, op);
}

cudaError_t launch_copy(const void* src, void* dst, size_t bytes, int grid, cudaStream_t stream)
{
    copy_kernel<<<grid, 512, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                          static_cast<long long>(bytes / 16));
    return cudaGetLastError();
}

}  // namespace qta

using namespace qta;

extern "C" {

size_t qta_codes_bytes(const qta_desc* d)
{
    if (check_desc(d) != QTA_OK) return 0;
    const size_t n = static_cast<size_t>(n_elems(d));
    return d->scheme == QTA_INT4_ASYM_G128 ? n / 2 : n;
}

size_t qta_scales_bytes(const qta_desc* d)
{
    if (check_desc(d) != QTA_OK) return 0;
    const size_t nb = static_cast<size_t>(n_elems(d)) / d->block;
    if (d->scheme == QTA_TACO_FP8) return nb;
    if (d->scheme == QTA_INT8_SYM_B64) return nb * 4;
    return nb * 2;
}

size_t qta_zeros_bytes(const qta_desc* d)
{
    if (check_desc(d) != QTA_OK) return 0;
    if (d->scheme != QTA_INT4_ASYM_G128 && d->scheme != QTA_INT8_ASYM_G128) return 0;
    return static_cast<size_t>(n_elems(d)) / d->block * 2;
}

size_t qta_state_bytes(const qta_desc* d)
{
    if (check_desc(d) != QTA_OK) return 0;
    return d->scheme == QTA_TACO_FP8 ? static_cast<size_t>(d->batch) * 2 * sizeof(float) : 0;
}

static qta_status compress_impl(const qta_desc* d, const void* x, int32_t x_dtype, const qta_qtensor* out,
                                int32_t mode, qta_stream_t stream)
{
    qta_status st = check_desc(d);
    if (st != QTA_OK) return st;
    if (x_dtype != QTA_BF16 && x_dtype != QTA_FP16 && x_dtype != QTA_FP32) return QTA_ERR_UNSUPPORTED;
    const int base_mode = mode & ~QTA_SCALE_ROUND_UP;
    if (d->scheme == QTA_TACO_FP8 && base_mode != QTA_SCALE_DELAYED && base_mode != QTA_SCALE_CURRENT)
        return QTA_ERR_INVALID_ARG;
    if (n_elems(d) == 0) return QTA_OK;
    if (!x) return QTA_ERR_INVALID_ARG;
    if (!aligned(x, 16)) return QTA_ERR_ALIGNMENT;
    if ((st = check_qtensor(d, out)) != QTA_OK) return st;
    if (!encoder_ready()) return QTA_ERR_CUDA;
    int sms = 0, smem_sm = 0;
    unsigned int* err = nullptr;
    if (device_info(&sms, &smem_sm, &err) != cudaSuccess) return QTA_ERR_CUDA;

    const int64_t segs = n_elems(d) / 64;
    CompressParams p;
    std::memset(&p, 0, sizeof(p));
    if (!map_values(&p.in_map, x_dtype, x, segs)) return QTA_ERR_CUDA;
    if (!map_codes(&p.out_map, d->scheme, out->codes, segs)) return QTA_ERR_CUDA;
    p.scales = out->scales;
    p.zeros = out->zeros;
    p.state = out->state;
    p.err = err;
    p.M = static_cast<int>(segs);
    p.n_warp_tiles = static_cast<int>((segs + 31) / 32);
    p.lanes_per_block = lanes_of(d);
    p.lanes_log2 = log2i(p.lanes_per_block);
    p.seg_per_tensor = make_fastdiv(static_cast<uint32_t>(d->rows * d->cols / 64));
    p.round_up = (mode & QTA_SCALE_ROUND_UP) ? 1 : 0;
    p.chan = out->chan;
    p.seg_per_row = make_fastdiv(static_cast<uint32_t>(d->cols / 64));
    const int sch = d->scheme;  // qta_scheme values equal the kernel scheme kinds
    const int chan_bytes = static_cast<int>(d->cols) * 4;
    p.chan_smem = (out->chan && compress_smem(x_dtype, sch) + chan_bytes <= smem_optin()) ? 1 : 0;
    const int grid = grid_for(p.n_warp_tiles, compress_warps(x_dtype), sms, d->max_sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (d->scheme == QTA_TACO_FP8 && base_mode == QTA_SCALE_CURRENT) {
        cudaError_t e = launch_state(out->state, d->batch, STATE_RESET_AMAX, s);
        if (e == cudaSuccess) e = launch_compress(x_dtype, sch, true, p, grid, s);
        if (e == cudaSuccess) e = launch_state(out->state, d->batch, STATE_SET_SCALE, s);
        if (e != cudaSuccess) return QTA_ERR_CUDA;
    }
    return cuda_status(launch_compress(x_dtype, sch, false, p, grid, s));
}

qta_status taco_compress(const qta_desc* d, const void* x, int32_t x_dtype, const qta_qtensor* out, int32_t mode,
                         qta_stream_t stream)
{
    return compress_impl(d, x, x_dtype, out, mode, stream);
}

qta_status qar_requant(const qta_desc* d, const float* sum, const qta_qtensor* out, int32_t mode,
                       qta_stream_t stream)
{
    return compress_impl(d, sum, QTA_FP32, out, mode, stream);
}

qta_status taco_decompress(const qta_desc* d, const qta_qtensor* in, void* y, int32_t y_dtype, qta_stream_t stream)
{
    qta_status st = check_desc(d);
    if (st != QTA_OK) return st;
    if (y_dtype != QTA_BF16 && y_dtype != QTA_FP16 && y_dtype != QTA_FP32) return QTA_ERR_UNSUPPORTED;
    if (n_elems(d) == 0) return QTA_OK;
    if (!y) return QTA_ERR_INVALID_ARG;
    if (!aligned(y, 16)) return QTA_ERR_ALIGNMENT;
    if ((st = check_qtensor(d, in)) != QTA_OK) return st;
    if (!encoder_ready()) return QTA_ERR_CUDA;
    int sms = 0, smem_sm = 0;
    unsigned int* err = nullptr;
    if (device_info(&sms, &smem_sm, &err) != cudaSuccess) return QTA_ERR_CUDA;

    const int64_t segs = n_elems(d) / 64;
    DecompressParams p;
    std::memset(&p, 0, sizeof(p));
    if (!map_codes(&p.in_map, d->scheme, in->codes, segs)) return QTA_ERR_CUDA;
    if (!map_values(&p.out_map, y_dtype, y, segs)) return QTA_ERR_CUDA;
    p.scales = in->scales;
    p.zeros = in->zeros;
    p.state = in->state;
    p.err = err;
    p.M = static_cast<int>(segs);
    p.n_warp_tiles = static_cast<int>((segs + 31) / 32);
    p.lanes_per_block = lanes_of(d);
    p.lanes_log2 = log2i(p.lanes_per_block);
    p.inv_block = 1.0f / static_cast<float>(d->block);
    p.seg_per_tensor = make_fastdiv(static_cast<uint32_t>(d->rows * d->cols / 64));
    p.chan_up = in->chan ? in->chan + d->cols : nullptr;
    p.seg_per_row = make_fastdiv(static_cast<uint32_t>(d->cols / 64));
    const int chan_bytes = static_cast<int>(d->cols) * 4;
    p.chan_smem = (in->chan && decompress_smem(d->scheme, y_dtype) + chan_bytes <= smem_optin()) ? 1 : 0;
    const int grid = grid_for(p.n_warp_tiles, decompress_warps(y_dtype), sms, d->max_sms);
    return cuda_status(launch_decompress(d->scheme, y_dtype, p, grid, reinterpret_cast<cudaStream_t>(stream)));
}

// Shared argument checks and parameters of qar_reduce / qar_reduce_requant.
static qta_status reduce_params(const qta_desc* d, const qta_qtensor* shards, int32_t n_ranks, int64_t row_begin,
                                int64_t row_end, ReduceParams* p, int* sms, int* smem_sm, bool* empty)
{
    qta_status st = check_desc(d);
    if (st != QTA_OK) return st;
    if (d->batch != 1) return QTA_ERR_INVALID_ARG;
    if (n_ranks < 1) return QTA_ERR_INVALID_ARG;
    if (n_ranks > MAX_RANKS) return QTA_ERR_UNSUPPORTED;
    if (row_begin < 0 || row_end < row_begin || row_end > d->rows) return QTA_ERR_INVALID_ARG;
    if (!shards) return QTA_ERR_INVALID_ARG;
    *empty = (row_end == row_begin || d->cols == 0);
    if (*empty) return QTA_OK;
    for (int r = 0; r < n_ranks; ++r) {
        if ((st = check_qtensor(d, &shards[r])) != QTA_OK) return st;
        // one set of channel factors for every rank (the transform of the sum
        // is then the sum of the transforms)
        if (shards[r].chan != shards[0].chan) return QTA_ERR_INVALID_ARG;
    }
    return QTA_OK;
}

static qta_status reduce_fill(const qta_desc* d, const qta_qtensor* shards, int32_t n_ranks, int64_t row_begin,
                              int64_t row_end, ReduceParams* p, int* sms, int* smem_sm)
{
    if (!encoder_ready()) return QTA_ERR_CUDA;
    unsigned int* err = nullptr;
    if (device_info(sms, smem_sm, &err) != cudaSuccess) return QTA_ERR_CUDA;
    const int64_t segs = n_elems(d) / 64;
    const int64_t per_row = d->cols / 64;
    std::memset(p, 0, sizeof(*p));
    for (int r = 0; r < n_ranks; ++r) {
        const bool ok = (d->scheme == QTA_INT4_ASYM_G128)
                            ? map_codes4_rows64(&p->in_map[r], shards[r].codes, static_cast<uint64_t>(segs))
                            : map_codes(&p->in_map[r], d->scheme, shards[r].codes, segs);
        if (!ok) return QTA_ERR_CUDA;
        p->scales[r] = shards[r].scales;
        p->zeros[r] = shards[r].zeros;
        p->state[r] = shards[r].state;
    }
    const int64_t m_out = (row_end - row_begin) * per_row;
    p->err = err;
    p->n_ranks = n_ranks;
    p->seg_begin = static_cast<int>(row_begin * per_row);
    p->M_out = static_cast<int>(m_out);
    p->n_warp_tiles = static_cast<int>((m_out + 31) / 32);
    p->lanes_per_block = lanes_of(d);
    p->lanes_log2 = log2i(p->lanes_per_block);
    p->inv_block = 1.0f / static_cast<float>(d->block);
    p->chan_up = shards[0].chan ? shards[0].chan + d->cols : nullptr;
    p->seg_per_row = make_fastdiv(static_cast<uint32_t>(d->cols / 64));
    return QTA_OK;
}

qta_status qar_reduce_requant(const qta_desc* d, const qta_qtensor* shards, int32_t n_ranks, int64_t row_begin,
                              int64_t row_end, const qta_desc* od, const qta_qtensor* out, int32_t mode,
                              qta_stream_t stream)
{
    ReduceParams p;
    int sms = 0, smem_sm = 0;
    bool empty = false;
    qta_status st = reduce_params(d, shards, n_ranks, row_begin, row_end, &p, &sms, &smem_sm, &empty);
    if (st != QTA_OK) return st;
    if ((st = check_desc(od)) != QTA_OK) return st;
    if (od->cols != d->cols || od->batch * od->rows != row_end - row_begin) return QTA_ERR_INVALID_ARG;
    const int base_mode = mode & ~QTA_SCALE_ROUND_UP;
    if (od->scheme == QTA_TACO_FP8 && base_mode != QTA_SCALE_DELAYED && base_mode != QTA_SCALE_CURRENT)
        return QTA_ERR_INVALID_ARG;
    if (!reduce_requant_supported(d->scheme, od->scheme)) return QTA_ERR_UNSUPPORTED;
    if (empty) return QTA_OK;
    if ((st = check_qtensor(od, out)) != QTA_OK) return st;
    // the requantized sum keeps the shards' channel factors: with one set on
    // both sides the rescaling cancels between the reduce and the requant
    if (out->chan != shards[0].chan) return QTA_ERR_UNSUPPORTED;
    if ((st = reduce_fill(d, shards, n_ranks, row_begin, row_end, &p, &sms, &smem_sm)) != QTA_OK) return st;
    p.chan_up = nullptr;
    if (!map_codes(&p.out_map, od->scheme, out->codes, static_cast<uint64_t>(p.M_out))) return QTA_ERR_CUDA;
    p.q_scales = out->scales;
    p.q_zeros = out->zeros;
    p.q_state = out->state;
    p.q_lanes_per_block = lanes_of(od);
    p.q_lanes_log2 = log2i(p.q_lanes_per_block);
    p.q_seg_per_tensor = make_fastdiv(static_cast<uint32_t>(od->rows * od->cols / 64));
    p.q_round_up = (mode & QTA_SCALE_ROUND_UP) ? 1 : 0;
    const int grid = grid_for(p.n_warp_tiles, reduce_warps(), sms, d->max_sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (od->scheme == QTA_TACO_FP8 && base_mode == QTA_SCALE_CURRENT) {
        cudaError_t e = launch_state(out->state, od->batch, STATE_RESET_AMAX, s);
        if (e == cudaSuccess) e = launch_reduce_requant(d->scheme, od->scheme, true, p, grid, s);
        if (e == cudaSuccess) e = launch_state(out->state, od->batch, STATE_SET_SCALE, s);
        if (e != cudaSuccess) return QTA_ERR_CUDA;
    }
    return cuda_status(launch_reduce_requant(d->scheme, od->scheme, false, p, grid, s));
}

qta_status qar_reduce(const qta_desc* d, const qta_qtensor* shards, int32_t n_ranks, int64_t row_begin,
                      int64_t row_end, float* sum_out, qta_stream_t stream)
{
    ReduceParams p;
    int sms = 0, smem_sm = 0;
    bool empty = false;
    qta_status st = reduce_params(d, shards, n_ranks, row_begin, row_end, &p, &sms, &smem_sm, &empty);
    if (st != QTA_OK || empty) return st;
    if (!sum_out) return QTA_ERR_INVALID_ARG;
    if (!aligned(sum_out, 16)) return QTA_ERR_ALIGNMENT;
    if ((st = reduce_fill(d, shards, n_ranks, row_begin, row_end, &p, &sms, &smem_sm)) != QTA_OK) return st;
    if (!map_f32(&p.out_map, sum_out, static_cast<uint64_t>(p.M_out))) return QTA_ERR_CUDA;
    const int chan_bytes = static_cast<int>(d->cols) * 4;
    p.chan_smem = (p.chan_up && reduce_smem(d->scheme, OUT_F32) + chan_bytes <= smem_optin()) ? 1 : 0;
    const int grid = grid_for(p.n_warp_tiles, reduce_warps(), sms, d->max_sms);
    return cuda_status(launch_reduce(d->scheme, p, grid, reinterpret_cast<cudaStream_t>(stream)));
}

// Shared implementation of qar_dequant_add (sum_out) and
// qar_dequant_add_requant (out).
static qta_status accum_impl(const qta_desc* d, const qta_qtensor* in, const void* x, int32_t x_dtype,
                             float* sum_out, const qta_qtensor* out, int32_t mode, qta_stream_t stream)
{
    qta_status st = check_desc(d);
    if (st != QTA_OK) return st;
    if (x_dtype != QTA_BF16 && x_dtype != QTA_FP16 && x_dtype != QTA_FP32) return QTA_ERR_UNSUPPORTED;
    const bool requant = out != nullptr;
    const int base_mode = mode & ~QTA_SCALE_ROUND_UP;
    if (requant && d->scheme == QTA_TACO_FP8 && base_mode != QTA_SCALE_DELAYED && base_mode != QTA_SCALE_CURRENT)
        return QTA_ERR_INVALID_ARG;
    if (n_elems(d) == 0) return QTA_OK;
    if (!x || (!requant && !sum_out)) return QTA_ERR_INVALID_ARG;
    if (!aligned(x, 16) || (!requant && !aligned(sum_out, 16))) return QTA_ERR_ALIGNMENT;
    if ((st = check_qtensor(d, in)) != QTA_OK) return st;
    if (requant && (st = check_qtensor(d, out)) != QTA_OK) return st;
    if (in->chan || (requant && out->chan)) return QTA_ERR_UNSUPPORTED;   // ring hops: no rescaling
    {   // the output may not overlap an input: the kernel reads and writes in one pass
        const size_t n = static_cast<size_t>(n_elems(d));
        const void* ins[5] = {x, in->codes, in->scales, in->zeros, in->state};
        const size_t in_n[5] = {n * dtype_bytes(x_dtype), qta_codes_bytes(d), qta_scales_bytes(d),
                                qta_zeros_bytes(d), qta_state_bytes(d)};
        const void* outs[4] = {sum_out, nullptr, nullptr, nullptr};
        size_t out_n[4] = {requant ? 0 : n * 4, 0, 0, 0};
        if (requant) {
            outs[0] = out->codes;
            outs[1] = out->scales;
            outs[2] = out->zeros;
            outs[3] = out->state;
            out_n[0] = qta_codes_bytes(d);
            out_n[1] = qta_scales_bytes(d);
            out_n[2] = qta_zeros_bytes(d);
            out_n[3] = qta_state_bytes(d);
        }
        for (int i = 0; i < 4; ++i)
            for (int j = 0; j < 5; ++j)
                if (overlaps(outs[i], out_n[i], ins[j], in_n[j])) return QTA_ERR_INVALID_ARG;
    }
    if (!encoder_ready()) return QTA_ERR_CUDA;
    int sms = 0, smem_sm = 0;
    unsigned int* err = nullptr;
    if (device_info(&sms, &smem_sm, &err) != cudaSuccess) return QTA_ERR_CUDA;

    const int64_t segs = n_elems(d) / 64;
    AccumParams p;
    std::memset(&p, 0, sizeof(p));
    if (!map_codes(&p.in_map, d->scheme, in->codes, segs)) return QTA_ERR_CUDA;
    if (!map_values(&p.x_map, x_dtype, x, segs)) return QTA_ERR_CUDA;
    if (requant ? !map_codes(&p.out_map, d->scheme, out->codes, segs) : !map_f32(&p.out_map, sum_out, segs))
        return QTA_ERR_CUDA;
    p.scales = in->scales;
    p.zeros = in->zeros;
    p.state = in->state;
    p.err = err;
    p.M = static_cast<int>(segs);
    p.n_warp_tiles = static_cast<int>((segs + 31) / 32);
    p.lanes_per_block = lanes_of(d);
    p.lanes_log2 = log2i(p.lanes_per_block);
    p.inv_block = 1.0f / static_cast<float>(d->block);
    p.seg_per_tensor = make_fastdiv(static_cast<uint32_t>(d->rows * d->cols / 64));
    if (requant) {
        p.q_scales = out->scales;
        p.q_zeros = out->zeros;
        p.q_state = out->state;
        p.round_up = (mode & QTA_SCALE_ROUND_UP) ? 1 : 0;
    }
    int a_warps = 0, a_smem = 0;
    accum_cfg(d->scheme, x_dtype, requant, a_warps, a_smem);
    const int grid = grid_for(p.n_warp_tiles, a_warps, sms, d->max_sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (requant && d->scheme == QTA_TACO_FP8 && base_mode == QTA_SCALE_CURRENT) {
        cudaError_t e = launch_state(out->state, d->batch, STATE_RESET_AMAX, s);
        if (e == cudaSuccess) e = launch_accum(d->scheme, x_dtype, true, true, p, grid, s);
        if (e == cudaSuccess) e = launch_state(out->state, d->batch, STATE_SET_SCALE, s);
        if (e != cudaSuccess) return QTA_ERR_CUDA;
    }
    return cuda_status(launch_accum(d->scheme, x_dtype, requant, false, p, grid, s));
}

qta_status qar_dequant_add(const qta_desc* d, const qta_qtensor* in, const void* x, int32_t x_dtype, float* sum_out,
                           qta_stream_t stream)
{
    return accum_impl(d, in, x, x_dtype, sum_out, nullptr, QTA_SCALE_DELAYED, stream);
}

qta_status qar_dequant_add_requant(const qta_desc* d, const qta_qtensor* in, const void* x, int32_t x_dtype,
                                   const qta_qtensor* out, int32_t mode, qta_stream_t stream)
{
    if (!out) return QTA_ERR_INVALID_ARG;
    return accum_impl(d, in, x, x_dtype, nullptr, out, mode, stream);
}

size_t qta_chan_bytes(int64_t cols) { return cols > 0 ? static_cast<size_t>(cols) * 3 * sizeof(float) : 0; }

qta_status taco_channel_amax(const qta_desc* d, const void* x, int32_t x_dtype, float* chan, qta_stream_t stream)
{
    qta_status st = check_desc(d);
    if (st != QTA_OK) return st;
    if (x_dtype != QTA_BF16 && x_dtype != QTA_FP16 && x_dtype != QTA_FP32) return QTA_ERR_UNSUPPORTED;
    if (n_elems(d) == 0) return QTA_OK;
    if (!x || !chan) return QTA_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(chan, 16)) return QTA_ERR_ALIGNMENT;
    if (overlaps(x, static_cast<size_t>(n_elems(d)) * dtype_bytes(x_dtype), chan, qta_chan_bytes(d->cols)))
        return QTA_ERR_INVALID_ARG;
    return cuda_status(launch_channel_amax(x, x_dtype, d->batch * d->rows, d->cols, chan + 2 * d->cols,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

qta_status taco_ash_update(float* chan, int64_t cols, qta_stream_t stream)
{
    if (cols <= 0) return cols == 0 ? QTA_OK : QTA_ERR_INVALID_ARG;
    if (!chan) return QTA_ERR_INVALID_ARG;
    if (!aligned(chan, 16)) return QTA_ERR_ALIGNMENT;
    return cuda_status(launch_ash_update(chan, cols, reinterpret_cast<cudaStream_t>(stream)));
}

qta_status qta_sq_error(const void* a, int32_t a_dtype, const float* b, int64_t n, double* out,
                        qta_stream_t stream)
{
    if (a_dtype != QTA_BF16 && a_dtype != QTA_FP16 && a_dtype != QTA_FP32) return QTA_ERR_UNSUPPORTED;
    if (n < 0 || !out) return QTA_ERR_INVALID_ARG;
    if (n > 0 && (!a || !b)) return QTA_ERR_INVALID_ARG;
    if (!aligned(out, 8) || !aligned(a, 4) || !aligned(b, 4)) return QTA_ERR_ALIGNMENT;
    int sms = 0, smem_sm = 0;
    unsigned int* err = nullptr;
    if (device_info(&sms, &smem_sm, &err) != cudaSuccess) return QTA_ERR_CUDA;
    const long long blocks = (n + 255) / 256;
    const int grid = static_cast<int>(blocks < 4LL * sms ? (blocks > 0 ? blocks : 1) : 4LL * sms);
    return cuda_status(launch_sq_error(a, a_dtype, b, n, out, grid, reinterpret_cast<cudaStream_t>(stream)));
}

qta_status qta_wait_self_test(int32_t complete, qta_stream_t stream)
{
    int sms = 0, smem_sm = 0;
    unsigned int* err = nullptr;
    if (device_info(&sms, &smem_sm, &err) != cudaSuccess) return QTA_ERR_CUDA;
    wait_self_test_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(complete ? 1 : 0, err);
    return cuda_status(cudaGetLastError());
}

qta_status taco_update_scale(float* state, int64_t n_tensors, qta_stream_t stream)
{
    if (n_tensors < 0) return QTA_ERR_INVALID_ARG;
    if (n_tensors == 0) return QTA_OK;
    if (!state) return QTA_ERR_INVALID_ARG;
    if (!aligned(state, 4)) return QTA_ERR_ALIGNMENT;
    return cuda_status(launch_state(state, n_tensors, STATE_UPDATE, reinterpret_cast<cudaStream_t>(stream)));
}

qta_status qta_copy(const void* src, void* dst, size_t bytes, qta_stream_t stream)
{
    if (bytes == 0) return QTA_OK;
    if (!src || !dst) return QTA_ERR_INVALID_ARG;
    if (!aligned(src, 16) || !aligned(dst, 16) || (bytes & 15)) return QTA_ERR_ALIGNMENT;
    int sms = 0, smem_sm = 0;
    unsigned int* err = nullptr;
    if (device_info(&sms, &smem_sm, &err) != cudaSuccess) return QTA_ERR_CUDA;
    return cuda_status(launch_copy(src, dst, bytes, sms * 4, reinterpret_cast<cudaStream_t>(stream)));
}

qta_status qta_device_error(uint32_t* flags, int32_t clear)
{
    if (!flags) return QTA_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return QTA_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_flags, sizeof(v)) != cudaSuccess) return QTA_ERR_CUDA;
    *flags = v;
    if (clear && v) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_error_flags, &z, sizeof(z)) != cudaSuccess) return QTA_ERR_CUDA;
    }
    return QTA_OK;
}

const char* qta_status_string(qta_status s)
{
    switch (s) {
    case QTA_OK: return "QTA_OK";
    case QTA_ERR_INVALID_ARG: return "QTA_ERR_INVALID_ARG";
    case QTA_ERR_ALIGNMENT: return "QTA_ERR_ALIGNMENT";
    case QTA_ERR_UNSUPPORTED: return "QTA_ERR_UNSUPPORTED";
    case QTA_ERR_CUDA: return "QTA_ERR_CUDA";
    default: return "QTA_ERR_UNKNOWN";
    }
}

}  // extern "C"
