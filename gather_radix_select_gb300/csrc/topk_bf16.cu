// topk_bf16.cu -- instantiations of the selection kernel for bf16 rows
// (one translation unit per element type so the two compile in parallel).
#include "topk_impl.cuh"

namespace sel {

cudaError_t launch_topk_bf16(int mode, int threads, bool gather, size_t smem, const TopkArgs &a, cudaStream_t s,
                            int64_t grid, bool query, int *blocks_per_sm)
{
    return launch_e<uint16_t>(mode, threads, gather, smem, a, s, grid, query, blocks_per_sm);
}

}  // namespace sel
