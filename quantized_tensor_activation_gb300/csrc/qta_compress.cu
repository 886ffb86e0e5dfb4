// qta_compress.cu -- instantiations and launcher of the compress kernels
// (taco_compress, qar_requant and the CURRENT-mode amax pre-pass).
#include "qta_launch.h"

namespace qta {

int compress_warps(int in_kind)
{
    return in_kind == IN_FP32 ? CompressCfg<IN_FP32, S_TACO>::WARPS : CompressCfg<IN_BF16, S_TACO>::WARPS;
}

int compress_smem(int in_kind, int scheme)
{
    const bool f32 = in_kind == IN_FP32;
    const bool a4 = scheme == S_ASYM4;
    if (f32) return a4 ? CompressCfg<IN_FP32, S_ASYM4>::SMEM : CompressCfg<IN_FP32, S_TACO>::SMEM;
    return a4 ? CompressCfg<IN_BF16, S_ASYM4>::SMEM : CompressCfg<IN_BF16, S_TACO>::SMEM;
}

template <int IN, int SCH, bool AMAX, int LG = -1, bool CH = false>
static cudaError_t launch_one(const CompressParams& p, int grid, cudaStream_t stream)
{
    using C = CompressCfg<IN, SCH>;
    static std::atomic<unsigned> done{0};
    auto fn = compress_kernel<IN, SCH, AMAX, LG, CH>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(fn), C::SMEM, &done);
    if (e != cudaSuccess) return e;
    const int extra = (CH && p.chan_smem) ? static_cast<int>(p.seg_per_row.d) * SEG * 4 : 0;
    static std::atomic<int> per_sm{0};
    const int g = persistent_grid(reinterpret_cast<const void*>(fn), C::WARPS * 32, C::SMEM + extra, grid,
                                  p.n_warp_tiles, C::WARPS, &per_sm);
    return launch_pdl(fn, dim3(g), dim3(C::WARPS * 32), C::SMEM + extra, stream, p);
}

// TACO with 4 lanes per block (B = 256) runs a kernel compiled for that
// block size: 83 against 92 us on an 8192 x 5120 x 4 bf16 input.  The same
// specialisation for 2 lanes (B = 128) ran slower than the kernel that reads
// the block size at run time (141 against 129 us on 8192 x 4096 x 8), so
// B = 64 and 128 keep the run-time kernel.
// With the adaptive rescaling (p.chan) a separate instantiation applies the
// channel factors, so that the kernels without them keep their registers.
template <int IN, bool AMAX>
static cudaError_t launch_taco(const CompressParams& p, int grid, cudaStream_t s)
{
    if (p.chan) {
        if (p.lanes_log2 == 2) return launch_one<IN, S_TACO, AMAX, 2, true>(p, grid, s);
        return launch_one<IN, S_TACO, AMAX, -1, true>(p, grid, s);
    }
    if (p.lanes_log2 == 2) return launch_one<IN, S_TACO, AMAX, 2>(p, grid, s);
    return launch_one<IN, S_TACO, AMAX, -1>(p, grid, s);
}

template <int IN>
static cudaError_t launch_in(int scheme, bool amax_only, const CompressParams& p, int grid, cudaStream_t s)
{
    switch (scheme) {
    case S_TACO: return amax_only ? launch_taco<IN, true>(p, grid, s) : launch_taco<IN, false>(p, grid, s);
    case S_INT8SYM: return launch_one<IN, S_INT8SYM, false>(p, grid, s);
    case S_ASYM4: return launch_one<IN, S_ASYM4, false>(p, grid, s);
    case S_ASYM8: return launch_one<IN, S_ASYM8, false>(p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_compress(int in_kind, int scheme, bool amax_only, const CompressParams& p, int grid,
                            cudaStream_t stream)
{
    switch (in_kind) {
    case IN_BF16: return launch_in<IN_BF16>(scheme, amax_only, p, grid, stream);
    case IN_FP16: return launch_in<IN_FP16>(scheme, amax_only, p, grid, stream);
    case IN_FP32: return launch_in<IN_FP32>(scheme, amax_only, p, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qta
