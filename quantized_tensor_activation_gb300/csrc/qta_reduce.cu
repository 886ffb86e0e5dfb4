// qta_reduce.cu -- instantiations and launchers of the dequantize-reduce
// kernels: qar_reduce (FP32 sum) and the fused qar_reduce_requant.
#include "qta_launch.h"

namespace qta {

int reduce_warps() { return ReduceCfg<S_TACO>::WARPS; }

int reduce_smem(int scheme, int out_scheme)
{
    if (out_scheme == OUT_F32) return scheme == S_ASYM4 ? ReduceCfg<S_ASYM4>::SMEM : ReduceCfg<S_TACO>::SMEM;
    switch (scheme * 4 + out_scheme) {
    case S_TACO * 4 + S_TACO: return ReduceCfg<S_TACO, S_TACO>::SMEM;
    case S_INT8SYM * 4 + S_INT8SYM: return ReduceCfg<S_INT8SYM, S_INT8SYM>::SMEM;
    case S_ASYM4 * 4 + S_ASYM8: return ReduceCfg<S_ASYM4, S_ASYM8>::SMEM;
    case S_ASYM8 * 4 + S_ASYM8: return ReduceCfg<S_ASYM8, S_ASYM8>::SMEM;
    default: return 0;
    }
}

bool reduce_requant_supported(int scheme, int out_scheme) { return reduce_smem(scheme, out_scheme) > 0 && out_scheme != OUT_F32; }

template <int SCH, int OSCH, bool AMAX, int LG = -1, bool CH = false, int NR = 0>
static cudaError_t launch_r(const ReduceParams& p, int grid, cudaStream_t stream)
{
    using C = ReduceCfg<SCH, OSCH, LG>;
    static std::atomic<unsigned> done{0};
    auto fn = reduce_kernel<SCH, OSCH, AMAX, LG, CH, NR>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(fn), C::SMEM, &done);
    if (e != cudaSuccess) return e;
    const int extra = (CH && p.chan_smem) ? static_cast<int>(p.seg_per_row.d) * SEG * 4 : 0;
    static std::atomic<int> per_sm{0};
    const int g = persistent_grid(reinterpret_cast<const void*>(fn), C::WARPS * 32, C::SMEM + extra, grid,
                                  p.n_warp_tiles, C::WARPS, &per_sm);
    return launch_pdl(fn, dim3(g), dim3(C::WARPS * 32), C::SMEM + extra, stream, p);
}

// The INT4 reduces (FP32 sum and fused) are also compiled for 4 and 8 shards:
// the rank loop unrolled, every shard index a constant (flash_int4's fused
// kernel 98.6 -> 84.5 us, its FP32 sum 103.0 -> 97.5 us).  Other counts run
// the kernel that reads the count at run time.  The TACO fused kernels compiled that way were slower (gpt_tp
// 60.5 -> 61.6 us, qwen_grad 43.3 -> 43.8 us) and the INT8 one no faster.
template <int SCH, int OSCH, bool AMAX, int LG = -1>
static cudaError_t launch_rn(const ReduceParams& p, int grid, cudaStream_t stream)
{
    switch (p.n_ranks) {
    case 4: return launch_r<SCH, OSCH, AMAX, LG, false, 4>(p, grid, stream);
    case 8: return launch_r<SCH, OSCH, AMAX, LG, false, 8>(p, grid, stream);
    default: return launch_r<SCH, OSCH, AMAX, LG>(p, grid, stream);
    }
}

cudaError_t launch_reduce(int scheme, const ReduceParams& p, int grid, cudaStream_t stream)
{
    switch (scheme) {
    case S_TACO:   // compiled per block size: the inverse transform's strips are constants
        if (p.chan_up) {   // the adaptive rescaling: its own instantiation
            switch (p.lanes_log2) {
            case 0: return launch_r<S_TACO, OUT_F32, false, 0, true>(p, grid, stream);
            case 1: return launch_r<S_TACO, OUT_F32, false, 1, true>(p, grid, stream);
            case 2: return launch_r<S_TACO, OUT_F32, false, 2, true>(p, grid, stream);
            default: return cudaErrorInvalidValue;
            }
        }
        switch (p.lanes_log2) {
        case 0: return launch_r<S_TACO, OUT_F32, false, 0>(p, grid, stream);
        case 1: return launch_r<S_TACO, OUT_F32, false, 1>(p, grid, stream);
        case 2: return launch_r<S_TACO, OUT_F32, false, 2>(p, grid, stream);
        default: return cudaErrorInvalidValue;
        }
    case S_INT8SYM: return launch_r<S_INT8SYM, OUT_F32, false>(p, grid, stream);
    case S_ASYM4: return launch_rn<S_ASYM4, OUT_F32, false>(p, grid, stream);
    case S_ASYM8: return launch_r<S_ASYM8, OUT_F32, false>(p, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_reduce_requant(int scheme, int out_scheme, bool amax_only, const ReduceParams& p, int grid,
                                  cudaStream_t stream)
{
    switch (scheme * 4 + out_scheme) {
    case S_TACO * 4 + S_TACO:
        // equal blocks of 4 lanes (B = 256, no transform): compiled for that
        // block size, 45.1 -> 43.6 us on 4 x 8192 x 5120, and with two ranks'
        // tiles per stage, 45.0 -> 44.2 us in the step; the same for 2 lanes
        // measured slower (59.6 -> 60.7 us on 8 x 8192 x 4096), and two ranks
        // per stage did not change it (60.5 us)
        if (p.q_lanes_log2 == 2 && p.lanes_log2 == 2)
            return amax_only ? launch_r<S_TACO, S_TACO, true, 2>(p, grid, stream)
                             : launch_r<S_TACO, S_TACO, false, 2>(p, grid, stream);
        return amax_only ? launch_r<S_TACO, S_TACO, true>(p, grid, stream)
                         : launch_r<S_TACO, S_TACO, false>(p, grid, stream);
    case S_INT8SYM * 4 + S_INT8SYM: return launch_r<S_INT8SYM, S_INT8SYM, false>(p, grid, stream);
    case S_ASYM4 * 4 + S_ASYM8: return launch_rn<S_ASYM4, S_ASYM8, false>(p, grid, stream);
    case S_ASYM8 * 4 + S_ASYM8: return launch_r<S_ASYM8, S_ASYM8, false>(p, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qta
