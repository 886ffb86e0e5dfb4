// qta_accum.cu -- instantiations and launcher of the ring-hop kernels
// (incoming partial sum + local tensor, FP32 out or requantized).
#include "qta_launch.h"

namespace qta {

// Warps and shared memory of the kernel that launch_accum runs (the grid is
// sized from them).
template <int XIN>
static void accum_cfg_x(int scheme, bool requant, int& warps, int& smem)
{
    if (!requant) {
        warps = AccumCfg<XIN, OUT_F32>::WARPS;
        smem = AccumCfg<XIN, OUT_F32>::SMEM;
        return;
    }
    switch (scheme) {
    case S_TACO: warps = AccumCfg<XIN, S_TACO>::WARPS; smem = AccumCfg<XIN, S_TACO>::SMEM; break;
    case S_INT8SYM: warps = AccumCfg<XIN, S_INT8SYM>::WARPS; smem = AccumCfg<XIN, S_INT8SYM>::SMEM; break;
    case S_ASYM4: warps = AccumCfg<XIN, S_ASYM4>::WARPS; smem = AccumCfg<XIN, S_ASYM4>::SMEM; break;
    default: warps = AccumCfg<XIN, S_ASYM8>::WARPS; smem = AccumCfg<XIN, S_ASYM8>::SMEM; break;
    }
}

void accum_cfg(int scheme, int x_kind, bool requant, int& warps, int& smem)
{
    if (x_kind == IN_FP32)
        accum_cfg_x<IN_FP32>(scheme, requant, warps, smem);
    else
        accum_cfg_x<IN_BF16>(scheme, requant, warps, smem);
}

template <int SCH, int XIN, int OSCH, bool AMAX_ONLY, int LG = -1>
static cudaError_t launch_a1(const AccumParams& p, int grid, cudaStream_t stream)
{
    using C = AccumCfg<XIN, OSCH>;
    static std::atomic<unsigned> done{0};
    auto fn = accum_kernel<SCH, XIN, OSCH, AMAX_ONLY, LG>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(fn), C::SMEM, &done);
    if (e != cudaSuccess) return e;
    static std::atomic<int> per_sm{0};
    const int g = persistent_grid(reinterpret_cast<const void*>(fn), C::WARPS * 32, C::SMEM, grid, p.n_warp_tiles,
                                  C::WARPS, &per_sm);
    return launch_pdl(fn, dim3(g), dim3(C::WARPS * 32), C::SMEM, stream, p);
}

template <int SCH, int XIN, int OSCH, bool AMAX_ONLY>
static cudaError_t launch_a(const AccumParams& p, int grid, cudaStream_t stream)
{
    if constexpr (SCH == S_TACO) {
        switch (p.lanes_log2) {
        case 0: return launch_a1<SCH, XIN, OSCH, AMAX_ONLY, 0>(p, grid, stream);
        case 1: return launch_a1<SCH, XIN, OSCH, AMAX_ONLY, 1>(p, grid, stream);
        case 2: return launch_a1<SCH, XIN, OSCH, AMAX_ONLY, 2>(p, grid, stream);
        default: return cudaErrorInvalidValue;
        }
    } else {
        return launch_a1<SCH, XIN, OSCH, AMAX_ONLY>(p, grid, stream);
    }
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
