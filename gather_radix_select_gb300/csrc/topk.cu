// topk.cu -- host-side dispatch of the selection kernel (kernels: topk_impl.cuh,
// instantiated per element type in topk_f32.cu and topk_bf16.cu).
#include <cstdint>

#include "sel_internal.h"

namespace sel {

cudaError_t launch_topk(int dtype, int mode, int threads, bool gather, size_t smem, const TopkArgs &a, int64_t grid,
                        cudaStream_t stream)
{
    return dtype == 0 ? launch_topk_f32(mode, threads, gather, smem, a, stream, grid, false, nullptr)
                      : launch_topk_bf16(mode, threads, gather, smem, a, stream, grid, false, nullptr);
}

int topk_blocks_per_sm(int dtype, int mode, int threads, bool gather, size_t smem)
{
    int blocks = 0;
    const cudaError_t e = dtype == 0 ? launch_topk_f32(mode, threads, gather, smem, TopkArgs{}, nullptr, 0, true, &blocks)
                                     : launch_topk_bf16(mode, threads, gather, smem, TopkArgs{}, nullptr, 0, true, &blocks);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return blocks;
}

size_t topk_smem_limit()
{
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    // leave room for the kernel's static shared memory (barriers, per-warp counters)
    return optin > 1024 ? static_cast<size_t>(optin) - 1024 : 0;
}

int device_sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace sel
