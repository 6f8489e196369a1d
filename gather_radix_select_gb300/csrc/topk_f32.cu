// topk_f32.cu -- instantiations of the selection kernel for fp32 rows
// (one translation unit per element type so the two compile in parallel).
#include "topk_impl.cuh"

namespace sel {

cudaError_t launch_topk_f32(int mode, int threads, bool gather, size_t smem, const TopkArgs &a, cudaStream_t s,
                            int64_t grid, bool query, int *blocks_per_sm)
{
    return launch_e<uint32_t>(mode, threads, gather, smem, a, s, grid, query, blocks_per_sm);
}

cudaError_t launch_wait_selftest(int32_t *err_flag, long long cycles, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 32, 0, s>>>(err_flag, cycles);
    return cudaGetLastError();
}

}  // namespace sel
