// qta_decompress.cu -- instantiations and launcher of the decompress kernels.
#include "qta_launch.h"

namespace qta {

int decompress_warps(int out_kind)
{
    return out_kind == IN_FP32 ? DecompressCfg<S_TACO, IN_FP32>::WARPS : DecompressCfg<S_TACO, IN_BF16>::WARPS;
}

int decompress_smem(int scheme, int out_kind)
{
    const bool f32 = out_kind == IN_FP32;
    const bool a4 = scheme == S_ASYM4;
    if (f32) return a4 ? DecompressCfg<S_ASYM4, IN_FP32>::SMEM : DecompressCfg<S_TACO, IN_FP32>::SMEM;
    return a4 ? DecompressCfg<S_ASYM4, IN_BF16>::SMEM : DecompressCfg<S_TACO, IN_BF16>::SMEM;
}


template <int SCH, int OUT, int LG = -1, bool CH = false>
static cudaError_t launch_d(const DecompressParams& p, int grid, cudaStream_t stream)
{
    using C = DecompressCfg<SCH, OUT>;
    static std::atomic<unsigned> done{0};
    auto fn = decompress_kernel<SCH, OUT, LG, CH>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(fn), C::SMEM, &done);
    if (e != cudaSuccess) return e;
    const int extra = (CH && p.chan_smem) ? static_cast<int>(p.seg_per_row.d) * SEG * 4 : 0;
    static std::atomic<int> per_sm{0};
    const int g = persistent_grid(reinterpret_cast<const void*>(fn), C::WARPS * 32, C::SMEM + extra, grid,
                                  p.n_warp_tiles, C::WARPS, &per_sm);
    return launch_pdl(fn, dim3(g), dim3(C::WARPS * 32), C::SMEM + extra, stream, p);
}

// TACO kernels are compiled per block size (1, 2 or 4 lanes per block).
template <int SCH, int OUT>
static cudaError_t launch_d_lanes(const DecompressParams& p, int grid, cudaStream_t s)
{
    if constexpr (SCH != S_TACO) {
        return launch_d<SCH, OUT>(p, grid, s);
    } else if (p.chan_up) {   // the adaptive rescaling: its own instantiation
        switch (p.lanes_log2) {
        case 0: return launch_d<SCH, OUT, 0, true>(p, grid, s);
        case 1: return launch_d<SCH, OUT, 1, true>(p, grid, s);
        case 2: return launch_d<SCH, OUT, 2, true>(p, grid, s);
        default: return cudaErrorInvalidValue;
        }
    } else {
        switch (p.lanes_log2) {
        case 0: return launch_d<SCH, OUT, 0>(p, grid, s);
        case 1: return launch_d<SCH, OUT, 1>(p, grid, s);
        case 2: return launch_d<SCH, OUT, 2>(p, grid, s);
        default: return cudaErrorInvalidValue;
        }
    }
}

template <int SCH>
static cudaError_t launch_d_out(int out_kind, const DecompressParams& p, int grid, cudaStream_t s)
{
    switch (out_kind) {
    case IN_BF16: return launch_d_lanes<SCH, IN_BF16>(p, grid, s);
    case IN_FP16: return launch_d_lanes<SCH, IN_FP16>(p, grid, s);
    case IN_FP32: return launch_d_lanes<SCH, IN_FP32>(p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decompress(int scheme, int out_kind, const DecompressParams& p, int grid, cudaStream_t stream)
{
    switch (scheme) {
    case S_TACO: return launch_d_out<S_TACO>(out_kind, p, grid, stream);
    case S_INT8SYM: return launch_d_out<S_INT8SYM>(out_kind, p, grid, stream);
    case S_ASYM4: return launch_d_out<S_ASYM4>(out_kind, p, grid, stream);
    case S_ASYM8: return launch_d_out<S_ASYM8>(out_kind, p, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qta
