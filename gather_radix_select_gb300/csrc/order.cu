// order.cu -- value-ordered output of a selection.
//
// "Speed up PyTorch TopK with DeepSelect", "Performance and advanced tips"
// (item 3): a row's results may be ordered by index or by value, each at a
// cost.  The selection kernels write every row in ascending column order;
// this kernel re-orders one row per CTA by value, largest first, equal values
// by column ascending, fills (index -1) last.  A NaN counts as larger than
// every number (NaNs among themselves by column); only short rows, which are
// not checked for NaN, can hold one in a defined selection.  The ranking is
// order_core.cuh's stable radix sort; the staged row kernel ranks its rows
// itself and needs no second launch.
#include <cstdint>
#include <type_traits>

#include "order_core.cuh"
#include "sel_internal.h"

namespace sel {
namespace {

using order::kEpt;
using order::kWarpItems;
constexpr int32_t kStatusInval = 1;  // SEL_EINVAL

// Copies the key rows of the ordered positions s_pos[0, ng) of one row to gather_out[row], NT threads,
// 16-byte loads (key rows are re-read across rows and stay in L2) and streaming stores (the output
// is written once).  A negative position reads key row 0; one at or past comp_len writes a zero row
// and SEL_EINVAL to err_flag.  Debug builds check every key row read against key_span.
template <int NT>
__device__ void gather_ordered(const OrderArgs &a, int64_t row, const int32_t *s_pos, int ng)
{
    constexpr int kUnroll = 4;
    const int64_t batch = row / a.rows_per_batch;
    const uint16_t *kb = a.key + batch * a.key_batch_stride;
    const int64_t kspan = a.key_span - batch * a.key_batch_stride;
    const int vpr = static_cast<int>(a.d >> 3);  // 16-byte vectors per key row
    const int vsh = (vpr & (vpr - 1)) == 0 ? __ffs(vpr) - 1 : -1;
    uint4 *ob = reinterpret_cast<uint4 *>(a.gather_out + row * a.n_gather * a.d);
    const int total = ng * vpr;
    for (int t0 = threadIdx.x; t0 < total; t0 += kUnroll * NT) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int t = t0 + u * NT;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (t < total) {
                const int jj = vsh >= 0 ? (t >> vsh) : t / vpr;
                int64_t p = s_pos[jj];
                if (p < 0) p = 0;
                if (p >= a.comp_len) {
                    if (a.err_flag) atomicCAS(a.err_flag, 0, kStatusInval);
                } else if (SEL_IN_BOUNDS(p * a.key_row_stride + a.d <= kspan, a.err_flag)) {
                    v[u] = __ldg(reinterpret_cast<const uint4 *>(kb + p * a.key_row_stride) + (t - jj * vpr));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int t = t0 + u * NT;
            if (t < total) __stcs(ob + t, v[u]);
        }
    }
}

// One CTA per row of NT threads (32..512, NT * 8 >= k; a compile-time count keeps every
// shared-memory address a base plus an immediate).  Shared memory: NT*8 columns, NT*8 value words,
// then value_rank's items and counters.
template <bool BF16, bool I64, int NT>
__global__ void __launch_bounds__(NT) value_order_kernel(const OrderArgs a)
{
    extern __shared__ __align__(16) unsigned char s_raw[];
    constexpr int nt = NT, n_items = NT * kEpt;
    const int k = a.k;
    int32_t *s_col = reinterpret_cast<int32_t *>(s_raw);
    uint32_t *s_val = reinterpret_cast<uint32_t *>(s_col + n_items);
    unsigned char *s_rank = reinterpret_cast<unsigned char *>(s_val + n_items);
    const int64_t row = blockIdx.x;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const char *xr = static_cast<const char *>(a.x) + row * a.x_stride * (BF16 ? 2 : 4);
    const uint32_t fill_bits = BF16 ? 0xff80u : 0xff800000u;

    // load: item e of this thread is position p = 256 warp + 32 e + lane (each warp instruction
    // reads 32 consecutive entries); every load is issued before the first is used
    const int wbase = warp * kWarpItems;
    int32_t col[kEpt];
    uint32_t v[kEpt];
#pragma unroll
    for (int e = 0; e < kEpt; ++e) {
        const int p = wbase + e * 32 + lane;
        col[e] = -1;
        v[e] = fill_bits;
        if (p < k) {
            col[e] = static_cast<int32_t>(I64 ? static_cast<const int64_t *>(a.out_idx)[row * a.out_idx_stride + p]
                                              : static_cast<const int32_t *>(a.out_idx)[row * a.out_idx_stride + p]);
            if (a.out_val)
                v[e] = BF16 ? static_cast<const uint16_t *>(a.out_val)[row * a.out_val_stride + p]
                            : static_cast<const uint32_t *>(a.out_val)[row * a.out_val_stride + p];
        }
    }
    if (!a.out_val) {
#pragma unroll
        for (int e = 0; e < kEpt; ++e)
            if (col[e] >= 0)
                v[e] = BF16 ? reinterpret_cast<const uint16_t *>(xr)[col[e]] : reinterpret_cast<const uint32_t *>(xr)[col[e]];
    }
    bool valid[kEpt];
#pragma unroll
    for (int e = 0; e < kEpt; ++e) {
        const int p = wbase + e * 32 + lane;
        valid[e] = col[e] >= 0;
        if (!valid[e]) v[e] = fill_bits;  // an entry with no column (a fill) keeps the fill value
        s_col[p] = col[e];
        s_val[p] = v[e];
    }
    order::value_rank<BF16, NT>(v, valid, s_rank);

    // write (coalesced): rank j's column and value, looked up by position; the first n_gather
    // columns also go to s_pos (value_rank's item words: free once every position is read)
    const int ng = static_cast<int>(a.n_gather);
    int32_t c_out[kEpt];
    uint32_t v_out[kEpt];
#pragma unroll
    for (int u = 0; u < kEpt; ++u) {
        const int j = t + u * nt;
        const int slot = j < k ? order::ranked_position<BF16>(s_rank, j) : 0;
        c_out[u] = s_col[slot];
        v_out[u] = s_val[slot];
    }
    int32_t *s_pos = reinterpret_cast<int32_t *>(s_rank);
    if (ng > 0) __syncthreads();  // every rank read before s_pos overwrites the items
#pragma unroll
    for (int u = 0; u < kEpt; ++u) {
        const int j = t + u * nt;
        if (j >= k) break;
        if (j < ng) s_pos[j] = c_out[u];
        if (I64)
            static_cast<int64_t *>(a.out_idx)[row * a.out_idx_stride + j] = c_out[u];
        else
            static_cast<int32_t *>(a.out_idx)[row * a.out_idx_stride + j] = c_out[u];
        if (a.out_val) {
            if (BF16)
                static_cast<uint16_t *>(a.out_val)[row * a.out_val_stride + j] = static_cast<uint16_t>(v_out[u]);
            else
                static_cast<uint32_t *>(a.out_val)[row * a.out_val_stride + j] = v_out[u];
        }
    }
    if (ng > 0) {
        __syncthreads();
        gather_ordered<NT>(a, row, s_pos, ng);
    }
}

template <bool BF16, bool I64, int NT>
cudaError_t launch_order(const OrderArgs &a, size_t smem, cudaStream_t stream)
{
    auto *kern = value_order_kernel<BF16, I64, NT>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    kern<<<static_cast<unsigned>(a.rows), NT, smem, stream>>>(a);
    return cudaGetLastError();
}

template <bool BF16, bool I64>
cudaError_t launch_nt(int threads, const OrderArgs &a, size_t smem, cudaStream_t stream)
{
    switch (threads) {
    case 32: return launch_order<BF16, I64, 32>(a, smem, stream);
    case 64: return launch_order<BF16, I64, 64>(a, smem, stream);
    case 128: return launch_order<BF16, I64, 128>(a, smem, stream);
    case 256: return launch_order<BF16, I64, 256>(a, smem, stream);
    case 512: return launch_order<BF16, I64, 512>(a, smem, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_value_order(int dtype, bool idx_i64, const OrderArgs &a_in, cudaStream_t stream)
{
    OrderArgs a = a_in;
    if (a.rows <= 0) return cudaSuccess;
    if (a.rows > 0x7fffffffLL || a.k < 1 || a.k > (1 << order::kSlotBits)) return cudaErrorInvalidValue;
    int threads = 32;  // a power of two from 32 to 512 with threads * 8 >= k
    while (threads * kEpt < a.k) threads <<= 1;
    const int n_items = threads * kEpt;
    const size_t smem = static_cast<size_t>(n_items) * (sizeof(int32_t) + sizeof(uint32_t)) +
                        (dtype == 1 ? order::rank_smem_bytes<true>(threads) : order::rank_smem_bytes<false>(threads));
    return dtype == 1 ? (idx_i64 ? launch_nt<true, true>(threads, a, smem, stream)
                                 : launch_nt<true, false>(threads, a, smem, stream))
                      : (idx_i64 ? launch_nt<false, true>(threads, a, smem, stream)
                                 : launch_nt<false, false>(threads, a, smem, stream));
}

}  // namespace sel
