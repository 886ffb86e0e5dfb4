// qta_accum.cu -- instantiations and launcher of the ring-hop kernels
// (incoming partial sum + local tensor, FP32 out or requantized).
#include "qta_launch.h"

namespace qta {

int accum_warps(int x_kind, bool requant)
{
    return requant ? (x_kind == IN_FP32 ? AccumCfg<IN_FP32, S_TACO>::WARPS : AccumCfg<IN_BF16, S_TACO>::WARPS)
                   : (x_kind == IN_FP32 ? AccumCfg<IN_FP32, OUT_F32>::WARPS : AccumCfg<IN_BF16, OUT_F32>::WARPS);
}

int accum_smem(int x_kind, bool requant)
{
    return requant ? (x_kind == IN_FP32 ? AccumCfg<IN_FP32, S_TACO>::SMEM : AccumCfg<IN_BF16, S_TACO>::SMEM)
                   : (x_kind == IN_FP32 ? AccumCfg<IN_FP32, OUT_F32>::SMEM : AccumCfg<IN_BF16, OUT_F32>::SMEM);
}

template <int SCH, int XIN, int OSCH, bool AMAX_ONLY>
static cudaError_t launch_a(const AccumParams& p, int grid, cudaStream_t stream)
{
    using C = AccumCfg<XIN, OSCH>;
    static std::atomic<unsigned> done{0};
    auto fn = accum_kernel<SCH, XIN, OSCH, AMAX_ONLY>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(fn), C::SMEM, &done);
    if (e != cudaSuccess) return e;
    return launch_pdl(fn, dim3(grid), dim3(C::WARPS * 32), C::SMEM, stream, p);
}

template <int SCH, int XIN>
static cudaError_t launch_a_mode(bool requant, bool amax_only, const AccumParams& p, int grid, cudaStream_t s)
{
    if (!requant) return launch_a<SCH, XIN, OUT_F32, false>(p, grid, s);
    if constexpr (SCH == S_TACO) {
        if (amax_only) return launch_a<SCH, XIN, SCH, true>(p, grid, s);
    }
    return launch_a<SCH, XIN, SCH, false>(p, grid, s);
}

template <int SCH>
static cudaError_t launch_a_x(int x_kind, bool requant, bool amax_only, const AccumParams& p, int grid,
                              cudaStream_t s)
{
    switch (x_kind) {
    case IN_BF16: return launch_a_mode<SCH, IN_BF16>(requant, amax_only, p, grid, s);
    case IN_FP16: return launch_a_mode<SCH, IN_FP16>(requant, amax_only, p, grid, s);
    case IN_FP32: return launch_a_mode<SCH, IN_FP32>(requant, amax_only, p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_accum(int scheme, int x_kind, bool requant, bool amax_only, const AccumParams& p, int grid,
                         cudaStream_t stream)
{
    switch (scheme) {
    case S_TACO: return launch_a_x<S_TACO>(x_kind, requant, amax_only, p, grid, stream);
    case S_INT8SYM: return launch_a_x<S_INT8SYM>(x_kind, requant, amax_only, p, grid, stream);
    case S_ASYM4: return launch_a_x<S_ASYM4>(x_kind, requant, amax_only, p, grid, stream);
    case S_ASYM8: return launch_a_x<S_ASYM8>(x_kind, requant, amax_only, p, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qta
