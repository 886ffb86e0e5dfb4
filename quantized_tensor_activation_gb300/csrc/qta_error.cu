// qta_error.cu -- squared-error reduction (reconstruction error of a codec
// round trip, for choosing the block size per tensor).
#include "qta_launch.h"

namespace qta {

template <int AK>
__device__ __forceinline__ double widen(const void* a, long long i)
{
    if constexpr (AK == IN_FP32) {
        return static_cast<double>(static_cast<const float*>(a)[i]);
    } else {
        const unsigned short h = static_cast<const unsigned short*>(a)[i];
        if constexpr (AK == IN_BF16)
            return static_cast<double>(__uint_as_float(static_cast<uint32_t>(h) << 16));
        else
            return static_cast<double>(__half2float(__ushort_as_half(h)));
    }
}

// out += sum over i of (a_i - b_i)^2 in FP64 (the difference of two values
// widened to FP64 is exact); one atomic add per block.
template <int AK>
__global__ void __launch_bounds__(256) sq_error_kernel(const void* __restrict__ a, const float* __restrict__ b,
                                                       long long n, double* out)
{
    double acc = 0.0;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n; i += stride) {
        const double d = widen<AK>(a, i) - static_cast<double>(__ldg(b + i));
        acc = fma(d, d, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    __shared__ double part[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) part[warp] = acc;
    __syncthreads();
    if (warp == 0) {
        acc = lane < static_cast<int>(blockDim.x >> 5) ? part[lane] : 0.0;
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) atomicAdd(out, acc);
    }
}

cudaError_t launch_sq_error(const void* a, int a_kind, const float* b, long long n, double* out, int grid,
                            cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(double), stream);
    if (e != cudaSuccess || n == 0) return e;
    switch (a_kind) {
    case IN_BF16: sq_error_kernel<IN_BF16><<<grid, 256, 0, stream>>>(a, b, n, out); break;
    case IN_FP16: sq_error_kernel<IN_FP16><<<grid, 256, 0, stream>>>(a, b, n, out); break;
    case IN_FP32: sq_error_kernel<IN_FP32><<<grid, 256, 0, stream>>>(a, b, n, out); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qta
