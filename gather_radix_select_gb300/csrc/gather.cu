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
// Debug builds check every key row read against kspan (elements from the batch base kb to the end
// of the key) and record SEL_EBOUNDS in err_flag instead of reading outside.
__device__ __forceinline__ void copy_rows(const uint16_t *kb, int64_t row_stride, int64_t d, uint16_t *out, int np,
                                          const int64_t *s_pos, int64_t kspan, int32_t *err_flag)
{
    const int vpr = static_cast<int>(d >> 3);  // 16-byte vectors per key row
    const int vsh = (vpr & (vpr - 1)) == 0 ? __ffs(vpr) - 1 : -1;  // log2(vpr), or -1
    uint4 *ob = reinterpret_cast<uint4 *>(out);
    const int total = np * vpr;
    if (vsh >= 1 && vpr <= 2 * kGatherThreads) {
        // rows of a power-of-two number (>= 2) of vectors: lpr = vpr / 2 lanes share a row and
        // thread t copies vectors c and c + lpr (c = t mod lpr) of rows t / lpr,
        // t / lpr + threads / lpr, ... -- no per-vector index division, each instruction covers
        // whole 128-byte pieces of the rows
        const int lsh = vsh - 1, lpr = vpr >> 1;
        const int c = static_cast<int>(threadIdx.x) & (lpr - 1);
        const int rstep = kGatherThreads >> lsh;
        constexpr int UR = kUnroll / 2;  // rows a thread has in flight (two vectors each)
        for (int jb = static_cast<int>(threadIdx.x) >> lsh; jb < np; jb += UR * rstep) {
            uint4 v[UR][2];
#pragma unroll
            for (int u = 0; u < UR; ++u) {
                const int jj = jb + u * rstep;
                v[u][0] = v[u][1] = make_uint4(0u, 0u, 0u, 0u);
                if (jj < np) {
                    const int64_t p = s_pos[jj];
                    if (p >= 0 && SEL_IN_BOUNDS(p * row_stride + d <= kspan, err_flag)) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(kb + p * row_stride) + c;
                        v[u][0] = __ldg(src);
                        v[u][1] = __ldg(src + lpr);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < UR; ++u) {
                const int jj = jb + u * rstep;
                if (jj < np) {
                    uint4 *dst = ob + (static_cast<int64_t>(jj) << vsh) + c;
                    __stcs(dst, v[u][0]);
                    __stcs(dst + lpr, v[u][1]);
                }
            }
        }
        return;
    }
    for (int t0 = threadIdx.x; t0 < total; t0 += kUnroll * kGatherThreads) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int t = t0 + u * kGatherThreads;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (t < total) {
                const int jj = vsh >= 0 ? (t >> vsh) : t / vpr;
                const int64_t p = s_pos[jj];
                if (p >= 0 && SEL_IN_BOUNDS(p * row_stride + d <= kspan, err_flag))
                    v[u] = __ldg(reinterpret_cast<const uint4 *>(kb + p * row_stride) + (t - jj * vpr));
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
    copy_rows(a.key + batch * a.key_batch_stride, a.key_row_stride, a.d, a.out + (row * a.n + j0) * a.d, np, s_pos,
              a.key_span - batch * a.key_batch_stride, a.err_flag);
    if (a.out2)
        copy_rows(a.key2 + batch * a.key2_batch_stride, a.key2_row_stride, a.d2, a.out2 + (row * a.n + j0) * a.d2, np,
                  s_pos, a.key2_span - batch * a.key2_batch_stride, a.err_flag);
}

// Order-preserving key of a score (larger value => larger key; -0 and +0 equal).
__device__ __forceinline__ uint32_t score_key(uint32_t u, bool bf16)
{
    if (bf16) {
        u = (u == 0x8000u) ? 0u : u;
        return (u & 0x8000u) ? (~u & 0xffffu) : (u | 0x8000u);
    }
    u = (u == 0x80000000u) ? 0u : u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ bool score_is_nan(uint32_t u, bool bf16)
{
    return bf16 ? (u & 0x7fffu) > 0x7f80u : (u & 0x7fffffffu) > 0x7f800000u;
}

// The row's block selection done in the CTA (n_blocks <= kBlockSelectMax): block c is chosen when
// fewer than topk_blocks candidates beat it (a larger key, or an equal key and a smaller index);
// the chosen ids are compacted in ascending order into s_blk, -1 after them.  A row with more
// candidates than topk_blocks holding a NaN sets nan_flag (its selection is then unspecified).
__device__ void select_blocks(const BlockArgs &a, int64_t row, int64_t n_cand, int32_t *s_blk)
{
    __shared__ uint32_t s_key[kBlockSelectMax];
    __shared__ int s_warp_cnt[kBlockSelectMax / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int nb = static_cast<int>(a.n_blocks), nc = static_cast<int>(n_cand), tb = a.topk_blocks;
    const bool bf16 = a.scores_bf16 != 0;
    bool nan = false;
    if (t < nb) {
        const uint32_t u = bf16 ? static_cast<const uint16_t *>(a.scores)[row * a.scores_stride + t]
                                : static_cast<const uint32_t *>(a.scores)[row * a.scores_stride + t];
        s_key[t] = score_key(u, bf16);
        nan = t < nc && score_is_nan(u, bf16);
    }
    if (__syncthreads_or(nan) && nc > tb && t == 0 && a.nan_flag) atomicOr(a.nan_flag, 1);
    bool chosen = false;
    if (t < nc) {
        const uint32_t kt = s_key[t];
        int beaten = 0;
        for (int i = 0; i < nc; ++i) {
            const uint32_t ki = s_key[i];
            beaten += (ki > kt) | ((ki == kt) & (i < t));
        }
        chosen = beaten < tb;
    }
    // ordered compaction; the first kBlockSelectMax threads are whole warps
    unsigned m = 0;
    if (t < kBlockSelectMax) {
        m = __ballot_sync(0xffffffffu, chosen);
        if (lane == 0) s_warp_cnt[warp] = __popc(m);
    }
    __syncthreads();
    if (t < kBlockSelectMax) {
        int base = 0, total = 0;
        for (int w = 0; w < kBlockSelectMax / 32; ++w) {
            base += w < warp ? s_warp_cnt[w] : 0;
            total += s_warp_cnt[w];
        }
        if (chosen) s_blk[base + __popc(m & ((1u << lane) - 1u))] = t;
        for (int j = total + t; j < tb; j += kBlockSelectMax) s_blk[j] = -1;
    }
}

// One CTA per row: the row's selected block ids (ascending; -1 fills last) are read into shared
// memory (or chosen here, see select_blocks), then every block expands to its positions blk * block_size + i, positions at or past the
// row's end become -1, and the valid positions are written first (ascending), -1 after them; the
// key rows of each chunk of positions are gathered as in gather_kernel (a -1 reads position 0).
__global__ void __launch_bounds__(kGatherThreads) block_expand_kernel(const BlockArgs a)
{
    extern __shared__ int32_t s_blk[];  // topk_blocks ids
    __shared__ int64_t s_pos[kPairsPerCta];
    const int64_t row = blockIdx.x / a.ctas_per_row;
    const int part = static_cast<int>(blockIdx.x - row * a.ctas_per_row);
    int32_t *prow = a.pos + row * a.pos_stride;
    const int tb = a.topk_blocks;
    int64_t pe = a.pos_limit;
    if (a.pos_end) {
        const int64_t e = a.pos_end[row];
        pe = e < 0 ? 0 : (e > a.pos_limit ? a.pos_limit : e);
    }
    if (a.scores)
        select_blocks(a, row, (pe + a.block_size - 1) / a.block_size, s_blk);
    else
        for (int j = threadIdx.x; j < tb; j += kGatherThreads) s_blk[j] = prow[j];
    __syncthreads();  // every id is read before the row is overwritten
    // blocks are ascending and only the last valid block can reach past pe, so the valid positions
    // of block j start at j * block_size and the row is: valid positions, then -1
    const int64_t bs = a.block_size;
    const int64_t npos = static_cast<int64_t>(tb) * bs;
    const uint16_t *kb = a.key ? a.key + (row / a.rows_per_batch) * a.key_batch_stride : nullptr;
    // this CTA's positions: all of them, or one chunk of kPairsPerCta when the row is split
    const int64_t qb = a.ctas_per_row > 1 ? static_cast<int64_t>(part) * kPairsPerCta : 0;
    const int64_t qe = a.ctas_per_row > 1 ? min(npos, qb + kPairsPerCta) : npos;
    for (int64_t q0 = qb; q0 < qe; q0 += kPairsPerCta) {
        const int np = static_cast<int>(qe - q0 < kPairsPerCta ? qe - q0 : kPairsPerCta);
        for (int i = threadIdx.x; i < np; i += kGatherThreads) {
            const int64_t q = q0 + i;
            const int64_t j = q / bs;
            const int32_t blk = s_blk[j];
            int64_t p = blk < 0 ? -1 : static_cast<int64_t>(blk) * bs + (q - j * bs);
            if (p >= pe) p = -1;
            prow[q] = static_cast<int32_t>(p);
            int64_t g = p < 0 ? 0 : p;  // safe position
            if (g >= a.comp_len) {
                g = -1;  // out of range: a zero row and an error flag
                if (a.err_flag && kb) atomicCAS(a.err_flag, 0, kStatusInval);
            }
            s_pos[i] = g;
        }
        __syncthreads();
        if (kb)
            copy_rows(kb, a.key_row_stride, a.d, a.out + (row * npos + q0) * a.d, np, s_pos,
                      a.key_span - (row / a.rows_per_batch) * a.key_batch_stride, a.err_flag);
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_block_expand(const BlockArgs &a_in, cudaStream_t stream)
{
    BlockArgs a = a_in;
    if (a.rows <= 0) return cudaSuccess;
    if (a.topk_blocks < 1) return cudaErrorInvalidValue;
    // a row selected in the kernel is split into chunks of kPairsPerCta positions, one CTA each;
    // block ids read from pos are expanded in place, so such a row stays with one CTA
    const int64_t npos = static_cast<int64_t>(a.topk_blocks) * a.block_size;
    a.ctas_per_row = a.scores ? static_cast<int32_t>((npos + kPairsPerCta - 1) / kPairsPerCta) : 1;
    const int64_t grid = a.rows * a.ctas_per_row;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(a.topk_blocks) * sizeof(int32_t);
    block_expand_kernel<<<static_cast<unsigned>(grid), kGatherThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

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
