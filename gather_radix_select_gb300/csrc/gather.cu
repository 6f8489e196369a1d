// gather.cu -- flat row gather of selected key rows.
//
// MindSpore hyper-parallel pull request "perf/gather-index-select"
// (description): gathering key[batch, position] with two index tensors is
// replaced by one index_select over the batch-flattened key, the batch offset
// folded into the position (flat row = batch * comp_len + position), with
// clamped ("safe") positions.  Here:
//     out[r, j, :] = key[r / rows_per_batch, max(idx[r, j], 0), :]
// Every CTA owns a run of (row, position) pairs of one row, stages their
// positions in shared memory and streams whole key rows with 16-byte loads
// (key rows are re-read many times and stay in L2) and 16-byte streaming
// stores (the output is written once and never re-read here).
//
// The pair form serves the same pull request's Indexer KL loss, which gathers
// two keys of different widths (the index key and the attention key) at the
// same positions: one launch stages the positions once and fills both
// outputs.
#include <cstdint>

#include "sel_internal.h"

namespace sel {
namespace {

constexpr int kPairsPerCta = 256;
constexpr int kUnroll = 4;
constexpr int32_t kStatusInval = 1;

// Copies the key rows at positions s_pos[0, np) (batch base kb, rows of d elements) to the
// contiguous output rows at ob; a position of -1 yields a zero row.
__device__ __forceinline__ void copy_rows(const uint16_t *kb, int64_t row_stride, int64_t d, uint16_t *out, int np,
                                          const int64_t *s_pos)
{
    const int vpr = static_cast<int>(d >> 3);  // 16-byte vectors per key row
    const int vsh = (vpr & (vpr - 1)) == 0 ? __ffs(vpr) - 1 : -1;  // log2(vpr), or -1
    uint4 *ob = reinterpret_cast<uint4 *>(out);
    const int total = np * vpr;
    for (int t0 = threadIdx.x; t0 < total; t0 += kUnroll * kGatherThreads) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int t = t0 + u * kGatherThreads;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (t < total) {
                const int jj = vsh >= 0 ? (t >> vsh) : t / vpr;
                const int64_t p = s_pos[jj];
                if (p >= 0) v[u] = __ldg(reinterpret_cast<const uint4 *>(kb + p * row_stride) + (t - jj * vpr));
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int t = t0 + u * kGatherThreads;
            if (t < total) __stcs(ob + t, v[u]);
        }
    }
}

__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const GatherArgs a)
{
    __shared__ int64_t s_pos[kPairsPerCta];
    const int64_t cta = blockIdx.x;
    const int64_t row = cta / a.ctas_per_row;
    const int64_t j0 = (cta - row * a.ctas_per_row) * a.pairs_per_cta;
    const int64_t j1 = min(a.n, j0 + a.pairs_per_cta);
    if (j0 >= j1) return;
    const int np = static_cast<int>(j1 - j0);
    for (int i = threadIdx.x; i < np; i += kGatherThreads) {
        const int64_t off = row * a.idx_row_stride + j0 + i;
        int64_t p = a.idx_i64 ? static_cast<const int64_t *>(a.idx)[off]
                              : static_cast<int64_t>(static_cast<const int32_t *>(a.idx)[off]);
        if (p < 0) p = 0;
        if (p >= a.comp_len) {
            p = -1;  // out of range: a zero row and an error flag
            if (a.err_flag) atomicCAS(a.err_flag, 0, kStatusInval);
        }
        s_pos[i] = p;
    }
    __syncthreads();
    const int64_t batch = row / a.rows_per_batch;
    copy_rows(a.key + batch * a.key_batch_stride, a.key_row_stride, a.d, a.out + (row * a.n + j0) * a.d, np, s_pos);
    if (a.out2)
        copy_rows(a.key2 + batch * a.key2_batch_stride, a.key2_row_stride, a.d2, a.out2 + (row * a.n + j0) * a.d2, np,
                  s_pos);
}

}  // namespace

cudaError_t launch_gather(const GatherArgs &a_in, cudaStream_t stream)
{
    GatherArgs a = a_in;
    a.pairs_per_cta = kPairsPerCta;
    a.ctas_per_row = static_cast<int32_t>((a.n + kPairsPerCta - 1) / kPairsPerCta);
    const int64_t grid = a.rows * a.ctas_per_row;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    gather_kernel<<<static_cast<unsigned>(grid), kGatherThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sel
