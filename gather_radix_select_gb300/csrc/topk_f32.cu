// topk_f32.cu -- instantiations of the selection kernel for fp32 rows
// (one translation unit per element type so the two compile in parallel).
#include "topk_impl.cuh"

namespace sel {

cudaError_t launch_topk_f32(int threads, bool gather, int cluster, size_t smem, const TopkArgs &a, cudaStream_t s)
{
    return launch_e<uint32_t>(threads, gather, cluster, smem, a, s);
}

int topk_occupancy_f32(int threads, bool gather, int cluster, size_t smem)
{
    return occupancy_e<uint32_t>(threads, gather, cluster, smem);
}

}  // namespace sel
