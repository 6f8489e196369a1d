// topk_bf16.cu -- instantiations of the selection kernel for bf16 rows
// (one translation unit per element type so the two compile in parallel).
#include "topk_impl.cuh"

namespace sel {

cudaError_t launch_topk_bf16(int threads, bool gather, int cluster, size_t smem, const TopkArgs &a, cudaStream_t s)
{
    return launch_e<uint16_t>(threads, gather, cluster, smem, a, s);
}

int topk_occupancy_bf16(int threads, bool gather, int cluster, size_t smem)
{
    return occupancy_e<uint16_t>(threads, gather, cluster, smem);
}

}  // namespace sel
