// qta_launch.h -- host-side launchers of the codec kernels (internal).
#pragma once

#include <atomic>
#include <utility>

#include "qta_kernels.cuh"

namespace qta {

// Dynamic shared memory a kernel needs (bytes).
int compress_smem(int in_kind, int scheme);
int decompress_smem(int scheme, int out_kind);
int reduce_smem(int scheme, int out_scheme);   // out_scheme: OUT_F32 or the requant scheme
bool reduce_requant_supported(int scheme, int out_scheme);

// Warps per CTA of each kernel family.
int compress_warps(int in_kind);
int decompress_warps(int out_kind);
int reduce_warps();
void accum_cfg(int scheme, int x_kind, bool requant, int& warps, int& smem);

cudaError_t launch_compress(int in_kind, int scheme, bool amax_only, const CompressParams& p, int grid,
                            cudaStream_t stream);
cudaError_t launch_decompress(int scheme, int out_kind, const DecompressParams& p, int grid,
                              cudaStream_t stream);
cudaError_t launch_reduce(int scheme, const ReduceParams& p, int grid, cudaStream_t stream);
cudaError_t launch_reduce_requant(int scheme, int out_scheme, bool amax_only, const ReduceParams& p, int grid,
                                  cudaStream_t stream);
cudaError_t launch_accum(int scheme, int x_kind, bool requant, bool amax_only, const AccumParams& p, int grid,
                         cudaStream_t stream);
cudaError_t launch_state(float* state, long long n, int op, cudaStream_t stream);
cudaError_t launch_sq_error(const void* a, int a_kind, const float* b, long long n, double* out, int grid,
                            cudaStream_t stream);
cudaError_t launch_copy(const void* src, void* dst, size_t bytes, int grid, cudaStream_t stream);

// Launch with programmatic stream serialization (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Per-device one-time setting of the dynamic shared-memory limit of a kernel.
cudaError_t ensure_smem_attr(const void* func, int smem, std::atomic<unsigned>* done_mask);
int persistent_grid(const void* func, int threads, int smem, int grid_1, int n_warp_tiles, int warps,
                    std::atomic<int>* per_sm_cache);

}  // namespace qta
