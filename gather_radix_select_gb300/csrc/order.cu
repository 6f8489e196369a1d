// order.cu -- value-ordered output of a selection.
//
// "Speed up PyTorch TopK with DeepSelect", "Performance and advanced tips"
// (item 3): a row's results may be ordered by index or by value, each at a
// cost.  The selection kernels write every row in ascending column order;
// this kernel re-orders one row per CTA by value, largest first, equal values
// by column ascending, fills (index -1) last.  A NaN counts as larger than
// every number (NaNs among themselves by column); only short rows, which are
// not checked for NaN, can hold one in a defined selection.
//
// Because the row arrives in ascending column order, a STABLE sort by value
// alone yields the column tie-break.  The sort is a least-significant-digit
// radix sort on the inverted order-preserving key of each value (-0 folded
// onto +0, any NaN above every number), rebased to the row's smallest
// inverted key: the k values of a top-k row span a narrow range, so only the
// bits that differ are sorted (8-bit digits; at most 3 passes for a bf16
// row, about 4 for fp32 normal scores).  Fills take the key one
// above the range and so stay last.  Each item carries its slot (12 bits)
// beside the key; the column and value bits are looked up by slot at the end.
//
// Each pass ranks 8-bit digits: every warp ranks its 256 items with warp
// match (items of equal digit in a warp find one another, the lowest lane of
// each group advances that warp's counter for the digit), one block-wide
// exclusive scan turns the per-warp counts into digit-major, warp-minor bases
// (stable), and each item is scattered to its rank.  Items sit warp-striped:
// item e of lane l in warp w is position 256 w + 32 e + l, so positions and
// the ranking order agree.
#include <cstdint>
#include <type_traits>

#include "sel_internal.h"

namespace sel {
namespace {

constexpr int kEpt = 8;         // items a thread holds
constexpr int kSlotBits = 12;   // k <= 4096
constexpr int kRadixBits = 8;
constexpr int kDigits = 1 << kRadixBits;
constexpr int kWarpItems = 32 * kEpt;
constexpr int32_t kStatusInval = 1;  // SEL_EINVAL

// inverted order-preserving keys: larger value => smaller key; NaN smallest
__device__ __forceinline__ uint32_t inv_key_f32(uint32_t u)
{
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
    u = (u == 0x80000000u) ? 0u : u;
    return (u & 0x80000000u) ? u : ~(u | 0x80000000u);
}

__device__ __forceinline__ uint32_t inv_key_bf16(uint32_t h)
{
    if ((h & 0x7fffu) > 0x7f80u) return 0u;
    h = (h == 0x8000u) ? 0u : h;
    return ((h & 0x8000u) ? h : ~(h | 0x8000u)) & 0xffffu;
}

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

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
// shared-memory address a base plus an immediate).  Shared memory: NT*8 items (K), NT*8 columns,
// NT*8 value words, the per-warp digit counters [NT/32][256], then the digit bases [256].
// The s_red words hold the warps' key minima and maxima, then each pass's warp totals.
template <bool BF16, bool I64, int NT>
__global__ void __launch_bounds__(NT) value_order_kernel(const OrderArgs a)
{
    using K = typename std::conditional<BF16, uint32_t, uint64_t>::type;
    extern __shared__ __align__(16) unsigned char s_raw[];
    __shared__ uint32_t s_red[64];
    constexpr int nt = NT, n_items = NT * kEpt, nw = NT / 32;
    const int k = a.k;
    K *s_item = reinterpret_cast<K *>(s_raw);
    int32_t *s_col = reinterpret_cast<int32_t *>(s_item + n_items);
    uint32_t *s_val = reinterpret_cast<uint32_t *>(s_col + n_items);
    uint32_t *s_cnt = s_val + n_items;       // [nw][kDigits]: per-warp counts, then per-warp bases
    uint32_t *s_base = s_cnt + nw * kDigits;  // [kDigits]: digit totals, then exclusive digit bases
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
    uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
    for (int e = 0; e < kEpt; ++e) {
        const int p = wbase + e * 32 + lane;
        if (col[e] < 0) v[e] = fill_bits;  // an entry with no column (a fill) keeps the fill value
        s_col[p] = col[e];
        s_val[p] = v[e];
        if (col[e] >= 0) {
            const uint32_t kp = BF16 ? inv_key_bf16(v[e]) : inv_key_f32(v[e]);
            kmin = min(kmin, kp);
            kmax = max(kmax, kp);
        }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0) {
        s_red[warp] = kmin;
        s_red[32 + warp] = kmax;
    }
    __syncthreads();
    kmin = 0xffffffffu;
    kmax = 0u;
#pragma unroll
    for (int w = 0; w < nw; ++w) {
        kmin = min(kmin, s_red[w]);
        kmax = max(kmax, s_red[32 + w]);
    }
    // keys rebased to the row's range; fills one above it (no valid entry: everything is a fill)
    const uint64_t range = kmin <= kmax ? static_cast<uint64_t>(kmax - kmin) : 0ull;
    const uint64_t fill_key = range + 1;
    const int bits = 64 - __clzll(static_cast<long long>(fill_key));
    K item[kEpt];
#pragma unroll
    for (int e = 0; e < kEpt; ++e) {
        const uint32_t kp = BF16 ? inv_key_bf16(v[e]) : inv_key_f32(v[e]);
        const uint64_t kk = col[e] >= 0 ? static_cast<uint64_t>(kp - kmin) : fill_key;
        item[e] = (static_cast<K>(kk) << kSlotBits) | static_cast<K>(wbase + e * 32 + lane);
    }
    const uint32_t lt = lanemask_lt();
    uint32_t *wcnt = s_cnt + warp * kDigits;
    constexpr int dpt = kDigits >= nt ? kDigits / nt : 1;  // digits a thread scans

    for (int shift = kSlotBits; shift < kSlotBits + bits; shift += kRadixBits) {
        const int nb = min(kRadixBits, kSlotBits + bits - shift);  // digit bits that can be nonzero
        // this warp's counters (the previous pass read them before its closing barrier)
#pragma unroll
        for (int i = lane; i < kDigits; i += 32) wcnt[i] = 0u;
        // the lanes holding the same digit in each of the warp's 8 item rows: one ballot per bit
        uint32_t dg[kEpt], peers[kEpt];
#pragma unroll
        for (int e = 0; e < kEpt; ++e) {
            dg[e] = static_cast<uint32_t>(item[e] >> shift) & (kDigits - 1);
            peers[e] = 0xffffffffu;
        }
#pragma unroll
        for (int b = 0; b < kRadixBits; ++b) {
            if (b < nb) {
#pragma unroll
                for (int e = 0; e < kEpt; ++e) {
                    const bool one = (dg[e] >> b) & 1u;
                    const uint32_t m = __ballot_sync(0xffffffffu, one);
                    peers[e] &= one ? m : ~m;
                }
            }
        }
        __syncwarp();
        // rank among the warp's earlier items of the digit: row e's lowest lane of each digit
        // advances the warp's counter
        uint32_t rk[kEpt];
#pragma unroll
        for (int e = 0; e < kEpt; ++e) {
            const int leader = __ffs(peers[e]) - 1;
            uint32_t base = 0u;
            if (lane == leader) {
                base = wcnt[dg[e]];
                wcnt[dg[e]] = base + __popc(peers[e]);
            }
            __syncwarp();
            rk[e] = __shfl_sync(0xffffffffu, base, leader) + __popc(peers[e] & lt);
        }
        __syncthreads();  // every warp's counts are in; every read of s_item in this pass is done
        // digits [dpt t, dpt t + dpt) (threads past the digits hold none): exclusive over the warps
        // in place, then an exclusive scan of the digit totals over the block
        uint32_t tot[dpt], sum = 0u;
#pragma unroll
        for (int i = 0; i < dpt; ++i) {
            const int d = t * dpt + i;
            uint32_t run = 0u;
            if (d < kDigits) {
#pragma unroll
                for (int w = 0; w < nw; ++w) {
                    const uint32_t c = s_cnt[w * kDigits + d];
                    s_cnt[w * kDigits + d] = run;
                    run += c;
                }
            }
            tot[i] = run;
            sum += run;
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_red[warp] = incl;
        __syncthreads();
        uint32_t run = incl - sum;
#pragma unroll
        for (int w = 0; w < nw - 1; ++w)
            if (w < warp) run += s_red[w];
#pragma unroll
        for (int i = 0; i < dpt; ++i) {
            const int d = t * dpt + i;
            if (d < kDigits) s_base[d] = run;
            run += tot[i];
        }
        __syncthreads();
        // rank = the digit's base + this warp's base within the digit + the rank within the warp
#pragma unroll
        for (int e = 0; e < kEpt; ++e) s_item[s_base[dg[e]] + wcnt[dg[e]] + rk[e]] = item[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < kEpt; ++e) item[e] = s_item[wbase + e * 32 + lane];
    }

    // write (coalesced): rank j's column and value, looked up by slot (s_item is in rank order:
    // every call makes at least one pass, fill_key >= 1); the first n_gather columns also go to
    // s_pos (the counters' words: n_items of them, free after the last pass)
    int32_t *s_pos = reinterpret_cast<int32_t *>(s_cnt);
    const int ng = static_cast<int>(a.n_gather);
#pragma unroll
    for (int u = 0; u < kEpt; ++u) {
        const int j = t + u * nt;
        if (j >= k) break;
        const int slot = static_cast<int>(s_item[j] & ((K(1) << kSlotBits) - 1));
        const int32_t c_out = s_col[slot];
        const uint32_t v_out = s_val[slot];
        if (j < ng) s_pos[j] = c_out;
        if (I64)
            static_cast<int64_t *>(a.out_idx)[row * a.out_idx_stride + j] = c_out;
        else
            static_cast<int32_t *>(a.out_idx)[row * a.out_idx_stride + j] = c_out;
        if (a.out_val) {
            if (BF16)
                static_cast<uint16_t *>(a.out_val)[row * a.out_val_stride + j] = static_cast<uint16_t>(v_out);
            else
                static_cast<uint32_t *>(a.out_val)[row * a.out_val_stride + j] = v_out;
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
    if (a.rows > 0x7fffffffLL || a.k < 1 || a.k > (1 << kSlotBits)) return cudaErrorInvalidValue;
    int threads = 32;  // a power of two from 32 to 512 with threads * 8 >= k
    while (threads * kEpt < a.k) threads <<= 1;
    const int n_items = threads * kEpt;
    const size_t ksz = dtype == 1 ? sizeof(uint32_t) : sizeof(uint64_t);
    const int counters = kDigits * (threads / 32) + kDigits;
    const size_t smem = static_cast<size_t>(n_items) * (ksz + sizeof(int32_t) + sizeof(uint32_t)) +
                        static_cast<size_t>(counters) * sizeof(uint32_t);
    return dtype == 1 ? (idx_i64 ? launch_nt<true, true>(threads, a, smem, stream)
                                 : launch_nt<true, false>(threads, a, smem, stream))
                      : (idx_i64 ? launch_nt<false, true>(threads, a, smem, stream)
                                 : launch_nt<false, false>(threads, a, smem, stream));
}

}  // namespace sel
