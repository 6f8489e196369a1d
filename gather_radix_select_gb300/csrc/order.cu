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
// bits that differ are sorted (4-bit digits; e.g. 2 passes for a bf16 row on
// a few levels, about 7 for fp32 normal scores).  Fills take the key one
// above the range and so stay last.  Each item carries its slot (12 bits)
// beside the key; the column and value bits are looked up by slot at the end.
//
// One pass, with each thread holding 8 consecutive items: per-thread digit
// counts (packed 4-bit counters in a register), written digit-major to shared
// memory, one block-wide exclusive scan over them (digit-major, thread-minor:
// stable), then a scatter of every item to its rank.
#include <cstdint>
#include <type_traits>

#include "sel_internal.h"

namespace sel {
namespace {

constexpr int kEpt = 8;         // items a thread holds (4-bit counters: at most 8 per digit)
constexpr int kSlotBits = 12;   // k <= 4096
constexpr int kRadixBits = 4;
constexpr int kDigits = 1 << kRadixBits;

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

// Counter i of the digit-major counter array, padded so that a thread reading its own 16
// consecutive counters hits distinct banks.
__device__ __forceinline__ int cpad(int i) { return i + (i >> 4); }

// The 8 consecutive items of thread t, read as 16-byte vectors.
__device__ __forceinline__ void load_items(const uint32_t *s_item, int t, uint32_t (&item)[kEpt])
{
    const uint4 a = reinterpret_cast<const uint4 *>(s_item + t * kEpt)[0];
    const uint4 b = reinterpret_cast<const uint4 *>(s_item + t * kEpt)[1];
    item[0] = a.x, item[1] = a.y, item[2] = a.z, item[3] = a.w;
    item[4] = b.x, item[5] = b.y, item[6] = b.z, item[7] = b.w;
}

__device__ __forceinline__ void load_items(const uint64_t *s_item, int t, uint64_t (&item)[kEpt])
{
    const ulonglong2 *p = reinterpret_cast<const ulonglong2 *>(s_item + t * kEpt);
#pragma unroll
    for (int i = 0; i < kEpt / 2; ++i) {
        const ulonglong2 v = p[i];
        item[2 * i] = v.x;
        item[2 * i + 1] = v.y;
    }
}

// One CTA per row of NT threads (32..512, NT * 8 >= k; a compile-time count keeps every
// shared-memory address a base plus an immediate).  Shared memory: NT*8 items (K), NT*8 columns,
// NT*8 value words, then the padded counters.
template <bool BF16, bool I64, int NT>
__global__ void __launch_bounds__(NT) value_order_kernel(const OrderArgs a)
{
    using K = typename std::conditional<BF16, uint32_t, uint64_t>::type;
    extern __shared__ __align__(16) unsigned char s_raw[];
    __shared__ uint32_t s_red[64];
    constexpr int nt = NT, n_items = NT * kEpt;
    const int k = a.k;
    K *s_item = reinterpret_cast<K *>(s_raw);
    int32_t *s_col = reinterpret_cast<int32_t *>(s_item + n_items);
    uint32_t *s_val = reinterpret_cast<uint32_t *>(s_col + n_items);
    uint32_t *s_cnt = s_val + n_items;
    const int64_t row = blockIdx.x;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    constexpr int nw = NT / 32;
    const char *xr = static_cast<const char *>(a.x) + row * a.x_stride * (BF16 ? 2 : 4);
    const uint32_t fill_bits = BF16 ? 0xff80u : 0xff800000u;

    // load (coalesced): columns, value bits and the inverted keys of the row's entries
    uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll 4
    for (int u = 0; u < kEpt; ++u) {
        const int j = t + u * nt;
        int32_t col = -1;
        uint32_t v = fill_bits, kp = 0u;
        if (j < k) {
            col = static_cast<int32_t>(I64 ? static_cast<const int64_t *>(a.out_idx)[row * a.out_idx_stride + j]
                                           : static_cast<const int32_t *>(a.out_idx)[row * a.out_idx_stride + j]);
            if (col >= 0) {
                if (a.out_val)
                    v = BF16 ? static_cast<const uint16_t *>(a.out_val)[row * a.out_val_stride + j]
                             : static_cast<const uint32_t *>(a.out_val)[row * a.out_val_stride + j];
                else
                    v = BF16 ? reinterpret_cast<const uint16_t *>(xr)[col] : reinterpret_cast<const uint32_t *>(xr)[col];
                kp = BF16 ? inv_key_bf16(v) : inv_key_f32(v);
                kmin = min(kmin, kp);
                kmax = max(kmax, kp);
            }
        }
        s_item[j] = kp;
        s_col[j] = col;
        s_val[j] = v;
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
    for (int w = 0; w < nw; ++w) {
        kmin = min(kmin, s_red[w]);
        kmax = max(kmax, s_red[32 + w]);
    }
    // keys rebased to the row's range; fills one above it (no valid entry: everything is a fill)
    const uint64_t range = kmin <= kmax ? static_cast<uint64_t>(kmax - kmin) : 0ull;
    const uint64_t fill_key = range + 1;
    const int bits = 64 - __clzll(static_cast<long long>(fill_key));
    K item[kEpt];
    load_items(s_item, t, item);
    int32_t cols[kEpt];
    {
        const int4 c0 = reinterpret_cast<const int4 *>(s_col + t * kEpt)[0];
        const int4 c1 = reinterpret_cast<const int4 *>(s_col + t * kEpt)[1];
        cols[0] = c0.x, cols[1] = c0.y, cols[2] = c0.z, cols[3] = c0.w;
        cols[4] = c1.x, cols[5] = c1.y, cols[6] = c1.z, cols[7] = c1.w;
    }
#pragma unroll
    for (int e = 0; e < kEpt; ++e) {
        const uint64_t kk = cols[e] >= 0 ? static_cast<uint64_t>(static_cast<uint32_t>(item[e]) - kmin) : fill_key;
        item[e] = (static_cast<K>(kk) << kSlotBits) | static_cast<K>(t * kEpt + e);
    }

    for (int shift = kSlotBits; shift < kSlotBits + bits; shift += kRadixBits) {
        // this thread's digit counts
        uint64_t packed = 0;
#pragma unroll
        for (int e = 0; e < kEpt; ++e) packed += 1ull << (4 * (static_cast<int>(item[e] >> shift) & (kDigits - 1)));
        __syncthreads();  // the previous reads of s_red, s_cnt and s_item are done
#pragma unroll
        for (int d = 0; d < kDigits; ++d) s_cnt[cpad(d * nt + t)] = static_cast<uint32_t>(packed >> (4 * d)) & 0xfu;
        __syncthreads();
        // exclusive scan over the digit-major counters; thread t owns counters [16 t, 16 t + 16)
        uint32_t sum = 0;
#pragma unroll
        for (int i = 0; i < kDigits; ++i) sum += s_cnt[cpad(t * kDigits + i)];
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
        for (int i = 0; i < kDigits; ++i) {
            const uint32_t ci = s_cnt[cpad(t * kDigits + i)];
            s_cnt[cpad(t * kDigits + i)] = run;
            run += ci;
        }
        __syncthreads();
        // rank = the digit's base for this thread + the item's rank among the thread's items of that digit
        packed = 0;
#pragma unroll
        for (int e = 0; e < kEpt; ++e) {
            const int d = static_cast<int>(item[e] >> shift) & (kDigits - 1);
            s_item[s_cnt[cpad(d * nt + t)] + (static_cast<uint32_t>(packed >> (4 * d)) & 0xfu)] = item[e];
            packed += 1ull << (4 * d);
        }
        __syncthreads();
        load_items(s_item, t, item);
    }

    // write (coalesced): rank j's column and value, looked up by slot (s_item is in rank order:
    // every call makes at least one pass, fill_key >= 1)
#pragma unroll
    for (int u = 0; u < kEpt; ++u) {
        const int j = t + u * nt;
        if (j >= k) break;
        const int slot = static_cast<int>(s_item[j] & ((K(1) << kSlotBits) - 1));
        const int32_t col = s_col[slot];
        const uint32_t v = s_val[slot];
        if (I64)
            static_cast<int64_t *>(a.out_idx)[row * a.out_idx_stride + j] = col;
        else
            static_cast<int32_t *>(a.out_idx)[row * a.out_idx_stride + j] = col;
        if (a.out_val) {
            if (BF16)
                static_cast<uint16_t *>(a.out_val)[row * a.out_val_stride + j] = static_cast<uint16_t>(v);
            else
                static_cast<uint32_t *>(a.out_val)[row * a.out_val_stride + j] = v;
        }
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
    const int counters = kDigits * threads;
    const size_t smem = static_cast<size_t>(n_items) * (ksz + sizeof(int32_t) + sizeof(uint32_t)) +
                        static_cast<size_t>(counters + counters / 16) * sizeof(uint32_t);
    return dtype == 1 ? (idx_i64 ? launch_nt<true, true>(threads, a, smem, stream)
                                 : launch_nt<true, false>(threads, a, smem, stream))
                      : (idx_i64 ? launch_nt<false, true>(threads, a, smem, stream)
                                 : launch_nt<false, false>(threads, a, smem, stream));
}

}  // namespace sel
