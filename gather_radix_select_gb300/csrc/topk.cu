// topk.cu -- host-side dispatch of the selection kernel (kernels: topk_impl.cuh,
// instantiated per element type in topk_f32.cu and topk_bf16.cu).
#include <cstdint>

#include "sel_internal.h"

namespace sel {

cudaError_t launch_topk(int dtype, int threads, bool gather, int cluster, size_t smem, const TopkArgs &a,
                        cudaStream_t stream)
{
    return dtype == 0 ? launch_topk_f32(threads, gather, cluster, smem, a, stream)
                      : launch_topk_bf16(threads, gather, cluster, smem, a, stream);
}

int topk_max_active_clusters(int dtype, int threads, bool gather, int cluster, size_t smem)
{
    return dtype == 0 ? topk_occupancy_f32(threads, gather, cluster, smem)
                      : topk_occupancy_bf16(threads, gather, cluster, smem);
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
