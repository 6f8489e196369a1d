// topk_impl.cuh -- batched row-wise top-k by radix select, one row per CTA or per
// thread-block cluster, with an optional fused gather of the selected key rows.
//
// What is computed ("Speed up PyTorch TopK with DeepSelect": "Basic TopK
// usage", "Working with variable-length rows", "NaN handling"): for each row
// r with n = clamp(row_end[r], 0, cols) valid columns, the k largest values
// (ties: smaller column first), or, when n <= k, every valid column followed
// by fills (index -1, value -inf).  Rows with n > k are checked for NaN.
//
// How (GB300 design):
//   * A row is split into `slice`-element pieces, one per CTA of a cluster of
//     `cluster` CTAs (1 <= cluster <= 16).  Each CTA stages its piece into
//     shared memory with bulk async copies (cp.async.bulk, 16 KB chunks, one
//     mbarrier each) and builds the first digit histogram while later chunks
//     are still in flight: the row is read from HBM exactly once.
//   * Order-preserving key: fp32/bf16 bits -> unsigned key, larger float =>
//     larger key, -0 folded onto +0.
//   * Radix select over digits taken from the most significant end (e.g.
//     11/11/10 bits for fp32).  Histograms live in shared memory; each warp
//     aggregates equal digits with __match_any_sync so one atomicAdd per
//     distinct digit per warp reaches shared memory.  In a cluster the CTAs'
//     histograms are summed into CTA 0's shared memory through distributed
//     shared memory (red.shared::cluster) behind a hardware cluster barrier
//     -- no global scratch, no spin waits.
//   * A level stops early when the threshold bin holds exactly the number of
//     keys still needed.
//   * Compaction is ordered: every warp owns a contiguous segment of the
//     slice, segment bases come from exclusive scans (over warps, then over
//     the CTAs of the cluster, in column order), and inside a warp positions
//     come from warp scans.  Keys equal to the threshold are therefore taken
//     in column order (smaller index wins), deterministically, and every
//     row's output is in ascending column order -- sorted_index costs nothing.
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "sel_internal.h"

namespace sel {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr long long kWaitCycles = 4000000000LL;  // bound on any mbarrier wait (~2 s)
constexpr int32_t kStatusInval = 1;
constexpr int32_t kStatusTimeout = 5;

template <typename E>
struct Elem;

template <>
struct Elem<uint32_t> {  // fp32 bit patterns
    static constexpr int KB = 32;
    static constexpr int V = 4;  // elements per 16-byte vector
    static constexpr uint32_t kFill = 0xFF800000u;
    static __device__ __forceinline__ uint32_t key(uint32_t u)
    {
        u = (u == 0x80000000u) ? 0u : u;
        return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    static __device__ __forceinline__ bool is_nan(uint32_t u) { return (u & 0x7fffffffu) > 0x7f800000u; }
    static __device__ __forceinline__ void unpack(const uint4 &q, uint32_t (&e)[4])
    {
        e[0] = q.x;
        e[1] = q.y;
        e[2] = q.z;
        e[3] = q.w;
    }
};

template <>
struct Elem<uint16_t> {  // bf16 bit patterns
    static constexpr int KB = 16;
    static constexpr int V = 8;
    static constexpr uint16_t kFill = 0xFF80u;
    static __device__ __forceinline__ uint32_t key(uint16_t h)
    {
        uint32_t u = h;
        u = (u == 0x8000u) ? 0u : u;
        return (u & 0x8000u) ? (~u & 0xffffu) : (u | 0x8000u);
    }
    static __device__ __forceinline__ bool is_nan(uint16_t h) { return (h & 0x7fffu) > 0x7f80u; }
    static __device__ __forceinline__ void unpack(const uint4 &q, uint16_t (&e)[8])
    {
        e[0] = (uint16_t)(q.x & 0xffffu);
        e[1] = (uint16_t)(q.x >> 16);
        e[2] = (uint16_t)(q.y & 0xffffu);
        e[3] = (uint16_t)(q.y >> 16);
        e[4] = (uint16_t)(q.z & 0xffffu);
        e[5] = (uint16_t)(q.z >> 16);
        e[6] = (uint16_t)(q.w & 0xffffu);
        e[7] = (uint16_t)(q.w >> 16);
    }
};

__device__ __forceinline__ void set_err(int32_t *flag, int32_t code)
{
    if (flag) atomicCAS(flag, 0, code);
}

// Bounded wait on an mbarrier phase: after ~2 s the wait gives up, records
// a timeout in err_flag and lets the CTA run on (so cluster barriers stay matched).
__device__ __forceinline__ void wait_phase(uint64_t *bar, uint32_t parity, int32_t *err)
{
    constexpr uint32_t kSuspendNs = 100000;  // each try sleeps in hardware for up to 0.1 ms
    if (mbar_try_wait(bar, parity, kSuspendNs)) return;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity, kSuspendNs)) {
        if (clock64() - t0 > kWaitCycles) {
            set_err(err, kStatusTimeout);
            return;
        }
    }
}

// Shared-memory histogram increment.  `agg`: warp-aggregated (one atomicAdd per
// distinct digit per warp, via __match_any_sync; all 32 lanes must call), else
// one plain shared atomicAdd per valid lane.
__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t digit, bool valid, int lane, bool agg)
{
    if (agg) {
        const unsigned peers = __match_any_sync(kFull, valid ? digit : 0xffffffffu);
        if (valid && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(peers)));
    } else if (valid) {
        atomicAdd(&hist[digit], 1u);
    }
}

__device__ __forceinline__ uint32_t warp_exclusive_scan(uint32_t v, int lane, uint32_t &total)
{
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += y;
    }
    total = __shfl_sync(kFull, inc, 31);
    return inc - v;
}

__device__ __forceinline__ uint32_t take_from_ties(uint32_t need, uint32_t before, uint32_t count)
{
    if (before >= need) return 0u;
    const uint32_t left = need - before;
    return count < left ? count : left;
}

// Exclusive prefix sum over the CTA (thread order); `total` gets the CTA sum.
// Uses s_warp[NT/32]; contains two __syncthreads.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *s_warp, uint32_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const uint32_t t = s_warp[w];
        before += (w < warp) ? t : 0u;
        tot += t;
    }
    __syncthreads();
    total = tot;
    return before + inc - v;
}

// Threshold digit of a histogram h[0, nb): the digit d with
//   sum_{e > d} h[e] < need <= sum_{e >= d} h[e].
// Result in out[0] = d, out[1] = sum_{e > d} h[e], out[2] = h[d].  All threads call.
template <int NT>
__device__ void find_threshold(const uint32_t *h, int nb, uint32_t need, uint32_t *out, uint32_t *s_warp)
{
    const int tid = threadIdx.x;
    const int per = nb > NT ? nb / NT : 1;
    const int lo = tid * per;
    uint32_t s = 0;
    if (lo < nb)
        for (int i = 0; i < per; ++i) s += h[lo + i];
    // exclusive scan in reversed thread order gives the count above this thread's bins
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t inc = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(kFull, inc, o);
        if (lane + o < 32) inc += y;
    }
    if (lane == 0) s_warp[warp] = inc;
    __syncthreads();
    uint32_t above = inc - s;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) above += (w > warp) ? s_warp[w] : 0u;
    if (lo < nb && above < need && above + s >= need) {
        uint32_t acc = above;
        for (int i = per - 1; i >= 0; --i) {
            const uint32_t c = h[lo + i];
            if (acc + c >= need) {
                out[0] = static_cast<uint32_t>(lo + i);
                out[1] = acc;
                out[2] = c;
                break;
            }
            acc += c;
        }
    }
    __syncthreads();
}

__device__ __forceinline__ void store_idx(const TopkArgs &a, int64_t row, int64_t pos, int64_t col)
{
    if (!a.out_idx) return;
    if (a.idx_i64)
        static_cast<int64_t *>(a.out_idx)[row * a.out_idx_stride + pos] = col;
    else
        static_cast<int32_t *>(a.out_idx)[row * a.out_idx_stride + pos] = static_cast<int32_t>(col);
}

template <typename E>
__device__ __forceinline__ void store_val(const TopkArgs &a, int64_t row, int64_t pos, E v)
{
    static_cast<E *>(a.out_val)[row * a.out_val_stride + pos] = v;
}

// Copies key rows for output positions [j0, j1) of `row`:
//   gather_out[row, j, :] = key[row / rows_per_batch, max(col_j, 0), :]
// col_j = glist[j - j0] when glist is given, else j for j < n_short and 0 beyond.
template <int NT>
__device__ void gather_rows_of(const TopkArgs &a, int64_t row, int64_t j0, int64_t j1, const int32_t *glist,
                               int64_t n_short)
{
    const int vpr = static_cast<int>(a.d >> 3);  // 16-byte vectors per key row
    const int vsh = (vpr & (vpr - 1)) == 0 ? __ffs(vpr) - 1 : -1;  // log2(vpr), or -1
    const int64_t bb = row / a.rows_per_batch;
    const uint16_t *kb = a.key + bb * a.key_batch_stride;
    uint4 *ob = reinterpret_cast<uint4 *>(a.gather_out + (row * a.n_gather + j0) * a.d);
    const int total = static_cast<int>(j1 - j0) * vpr;
    constexpr int U = 4;
    for (int t0 = threadIdx.x; t0 < total; t0 += U * NT) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = t0 + u * NT;
            v[u] = make_uint4(0u, 0u, 0u, 0u);
            if (t < total) {
                const int jj = vsh >= 0 ? (t >> vsh) : t / vpr;
                const int64_t j = j0 + jj;
                int64_t p = glist ? static_cast<int64_t>(glist[jj]) : (j < n_short ? j : 0);
                if (p < 0) p = 0;
                if (p < a.comp_len)
                    v[u] = __ldg(reinterpret_cast<const uint4 *>(kb + p * a.key_row_stride) + (t - jj * vpr));
                else if (t - jj * vpr == 0)
                    set_err(a.err_flag, kStatusInval);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = t0 + u * NT;
            if (t < total) __stcs(ob + t, v[u]);
        }
    }
}

template <int NT>
struct MinBlocks {
    static constexpr int value = NT >= 512 ? 2 : (NT >= 256 ? 4 : 8);
};

template <typename E, int NT, bool CLUSTER, bool GATHER>
__global__ void __launch_bounds__(NT, MinBlocks<NT>::value) topk_kernel(const TopkArgs a)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    constexpr int W = NT / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t s_bar[kMaxChunks];
    __shared__ uint32_t s_warp[W];
    __shared__ uint32_t s_wgt[W], s_weq[W];
    __shared__ uint32_t s_wsel_base[W], s_weq_base[W];
    __shared__ uint32_t s_res[4];       // broadcast result of a histogram reduction
    __shared__ uint32_t s_all_g[kMaxCluster], s_all_e[kMaxCluster];  // per-CTA counts, written by the cluster
    __shared__ uint32_t s_cta_sel[2];   // (selected before this CTA, selected by this CTA)
    __shared__ uint32_t s_eq_before;    // keys of the threshold class before this CTA

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = CLUSTER ? cluster_rank() : 0u;
    const uint32_t csize = CLUSTER ? cluster_size() : 1u;
    const int64_t row = CLUSTER ? static_cast<int64_t>(cluster_id_x()) : static_cast<int64_t>(blockIdx.x);
    const bool agg = a.agg != 0;

    int64_t n = a.cols;
    if (a.row_end) {
        const int64_t re = a.row_end[row];
        n = re < 0 ? 0 : (re > a.cols ? a.cols : re);
    }
    const int k = a.k;
    const E *xrow = static_cast<const E *>(a.x) + row * a.stride;

    // ---------------------------------------------------------- short row
    if (n <= k) {  // the same decision in every CTA of the cluster
        const int per = (k + static_cast<int>(csize) - 1) / static_cast<int>(csize);
        const int j0 = static_cast<int>(rank) * per;
        const int j1 = min(k, j0 + per);
        for (int j = j0 + tid; j < j1; j += NT) {
            store_idx(a, row, j, j < n ? j : -1);
            if (a.want_values) store_val<E>(a, row, j, j < n ? xrow[j] : static_cast<E>(T::kFill));
        }
        if (GATHER) {
            const int64_t g1 = min(static_cast<int64_t>(j1), a.n_gather);
            if (j0 < g1) gather_rows_of<NT>(a, row, j0, g1, nullptr, n);
        }
        return;
    }

    // ------------------------------------------------- stage the slice
    E *buf = reinterpret_cast<E *>(smem);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + a.smem_hist_off);
    const int64_t lo = static_cast<int64_t>(rank) * a.slice;
    const int64_t hi = min(n, lo + a.slice);
    const int len = hi > lo ? static_cast<int>(hi - lo) : 0;
    const uint32_t bytes = static_cast<uint32_t>(len) * sizeof(E);
    const uint32_t bulk = bytes & ~15u;
    const int nchunks = static_cast<int>((bulk + kChunkBytes - 1) / kChunkBytes);
    // sampled first digit: only every sample_step-th 16-byte vector feeds the first histogram
    const bool sampled = a.sample_step > 1 && n >= 4LL * k && n >= static_cast<int64_t>(a.sample_min_cols);
    const int step = sampled ? a.sample_step : 1;

    if (tid == 0) {
        for (int c = 0; c < nchunks; ++c) mbar_init(&s_bar[c], 1);
        fence_mbar_init();
    }
    for (int i = tid; i < a.hist_bins; i += NT) hist[i] = 0u;
    __syncthreads();
    if (tid == 0) {
        const char *src = reinterpret_cast<const char *>(xrow + lo);
        for (int c = 0; c < nchunks; ++c) {
            const uint32_t nb = min(kChunkBytes, bulk - static_cast<uint32_t>(c) * kChunkBytes);
            mbar_arrive_expect_tx(&s_bar[c], nb);
            bulk_load(smem + static_cast<size_t>(c) * kChunkBytes, src + static_cast<size_t>(c) * kChunkBytes, nb,
                      &s_bar[c]);
        }
    }
    if (CLUSTER) cluster_sync();  // every CTA of the cluster has started before any remote access

    // -------------- first-digit histogram (every step-th vector) while chunks land
    const int sh0 = T::KB - a.bits[0];
    const int nb0 = 1 << a.bits[0];
    for (int c = 0; c < nchunks; ++c) {
        wait_phase(&s_bar[c], 0u, a.err_flag);
        const uint32_t cb = min(kChunkBytes, bulk - static_cast<uint32_t>(c) * kChunkBytes);
        const int nv = static_cast<int>(cb >> 4);
        const uint4 *vb = reinterpret_cast<const uint4 *>(smem + static_cast<size_t>(c) * kChunkBytes);
        for (int base = warp * 32; base * step < nv; base += NT) {
            const int v = (base + lane) * step;
            const bool ok = v < nv;
            E el[V];
            T::unpack(ok ? vb[v] : make_uint4(0u, 0u, 0u, 0u), el);
#pragma unroll
            for (int t = 0; t < V; ++t) hist_add(hist, T::key(el[t]) >> sh0, ok, lane, agg);
        }
    }
    {
        const int tail0 = static_cast<int>(bulk / sizeof(E));
        if (tid < len - tail0) {  // < 16 bytes left over: plain loads
            const E e = xrow[lo + tail0 + tid];
            buf[tail0 + tid] = e;
            if (!sampled) atomicAdd(&hist[T::key(e) >> sh0], 1u);
        }
    }
    __syncthreads();

    // Histogram reduction over the cluster: CTA 0's histogram is the merge target; CTA 0 evaluates
    // `decide` on the total and stores s_res[0..3] into every CTA.  Leaves every local histogram zero.
    auto reduce_decide = [&](int nb, auto &&decide) {
        if constexpr (CLUSTER) {
            if (rank != 0) {
                for (int i = tid; i < nb; i += NT) {
                    const uint32_t c = hist[i];
                    if (c) {
                        dsmem_add(map_to_rank(smem_addr(&hist[i]), 0u), c);
                        hist[i] = 0u;
                    }
                }
            }
            cluster_sync();
            if (rank == 0) {
                decide(hist, nb);  // block-wide; ends with __syncthreads
                for (int i = tid; i < nb; i += NT) hist[i] = 0u;
                if (tid < static_cast<int>(csize)) {
                    const uint32_t r = static_cast<uint32_t>(tid);
#pragma unroll
                    for (int w = 0; w < 4; ++w) dsmem_store(map_to_rank(smem_addr(&s_res[w]), r), s_res[w]);
                }
            }
            cluster_sync();
        } else {
            decide(hist, nb);
            for (int i = tid; i < nb; i += NT) hist[i] = 0u;
            __syncthreads();
        }
    };
    // exact threshold digit for `need` keys: s_res = {digit, count above it, count in it, 0}
    auto exact_threshold = [&](uint32_t need) {
        return [&, need](const uint32_t *h, int nb) {
            find_threshold<NT>(h, nb, need, s_res, s_warp);
            if (tid == 0) s_res[3] = 0u;
        };
    };

    // ---- candidate filter: mask byte per vector (bit t: key >= tkey), NaN check, ordered list
    uint16_t *list = reinterpret_cast<uint16_t *>(smem + a.smem_list_off);
    uint8_t *masks = smem + a.smem_mask_off;
    const int nvt = (len + V - 1) / V;  // 16-byte vectors in the slice (last one may be partial)
    const uint4 *vbuf = reinterpret_cast<const uint4 *>(buf);
    int L = 0;
    bool list_ok = false;
    auto build_list = [&](uint32_t tkey) {
        bool has_nan = false;
        for (int base = warp * 32; base < nvt; base += NT) {
            const int v = base + lane;
            if (v < nvt) {
                E el[V];
                T::unpack(vbuf[v], el);
                uint32_t m = 0;
#pragma unroll
                for (int t = 0; t < V; ++t) {
                    const bool in = v * V + t < len;
                    has_nan |= in && T::is_nan(el[t]);
                    m |= static_cast<uint32_t>(in && T::key(el[t]) >= tkey) << t;
                }
                masks[v] = static_cast<uint8_t>(m);
            }
        }
        if (__syncthreads_or(has_nan) && tid == 0 && a.nan_flag) atomicOr(a.nan_flag, 1);
        const int q = (nvt + NT - 1) / NT;
        const int v0 = min(nvt, tid * q), v1 = min(nvt, v0 + q);
        uint32_t c = 0;
        for (int v = v0; v < v1; ++v) c += __popc(static_cast<uint32_t>(masks[v]));
        uint32_t tot;
        uint32_t pos = block_exclusive_scan<NT>(c, s_warp, tot);
        list_ok = tot <= static_cast<uint32_t>(a.list_cap);
        if (list_ok) {
            for (int v = v0; v < v1; ++v) {
                uint32_t m = masks[v];
                while (m) {
                    const int b = __ffs(m) - 1;
                    list[pos++] = static_cast<uint16_t>(v * V + b);
                    m &= m - 1u;
                }
            }
        }
        L = list_ok ? static_cast<int>(tot) : 0;
        __syncthreads();
    };
    // histogram of the first digit over keys >= tkey (the list, or the whole slice when the list overflowed)
    auto candidate_hist = [&](uint32_t tkey) {
        if (list_ok) {
            for (int i = tid; i < L; i += NT) atomicAdd(&hist[T::key(buf[list[i]]) >> sh0], 1u);
        } else {
            for (int base = warp * 32; base < nvt; base += NT) {
                const int v = base + lane;
                if (v < nvt) {
                    E el[V];
                    T::unpack(vbuf[v], el);
#pragma unroll
                    for (int t = 0; t < V; ++t) {
                        const uint32_t kk = T::key(el[t]);
                        if (v * V + t < len && kk >= tkey) atomicAdd(&hist[kk >> sh0], 1u);
                    }
                }
            }
        }
        __syncthreads();
    };

    bool exact_done = false;
    if (sampled) {
        // threshold estimate from the sample: the highest digit that keeps, with a 4-sigma margin,
        // at least k keys of the whole row at or above it
        reduce_decide(nb0, [&](const uint32_t *h, int nb) {
            uint32_t s = 0;
            for (int i = tid; i < nb; i += NT) s += h[i];
            s = __reduce_add_sync(kFull, s);
            if (lane == 0) s_warp[warp] = s;
            __syncthreads();
            uint32_t total = 0;
#pragma unroll
            for (int w = 0; w < W; ++w) total += s_warp[w];
            __syncthreads();
            const float mu = static_cast<float>(k) * static_cast<float>(total) / static_cast<float>(n);
            const float want = mu + 4.0f * sqrtf(mu) + 2.0f;
            if (want >= static_cast<float>(total)) {
                if (tid == 0) {
                    s_res[0] = 0u;
                    s_res[3] = 0u;
                }
                __syncthreads();
            } else {
                find_threshold<NT>(h, nb, static_cast<uint32_t>(want), s_res, s_warp);
            }
        });
        const uint32_t tkey = s_res[0] << sh0;
        build_list(tkey);
        candidate_hist(tkey);
        // exact first digit among the candidates; flag 1 when fewer than k keys reached the estimate
        reduce_decide(nb0, [&](const uint32_t *h, int nb) {
            uint32_t s = 0;
            for (int i = tid; i < nb; i += NT) s += h[i];
            s = __reduce_add_sync(kFull, s);
            if (lane == 0) s_warp[warp] = s;
            __syncthreads();
            uint32_t total = 0;
#pragma unroll
            for (int w = 0; w < W; ++w) total += s_warp[w];
            __syncthreads();
            if (total < static_cast<uint32_t>(k)) {
                if (tid == 0) s_res[3] = 1u;
                __syncthreads();
            } else {
                find_threshold<NT>(h, nb, static_cast<uint32_t>(k), s_res, s_warp);
                if (tid == 0) s_res[3] = 0u;
                __syncthreads();
            }
        });
        exact_done = s_res[3] == 0u;
        if (!exact_done) {
            // the estimate was too high: exact histogram of the whole slice, then the list again
            list_ok = false;
            candidate_hist(0u);
        }
    }
    if (!exact_done) {
        reduce_decide(nb0, exact_threshold(static_cast<uint32_t>(k)));
        build_list(s_res[0] << sh0);
    }
    uint32_t prefix = s_res[0];  // selection class: (key >> shift) == prefix
    int shift = sh0;
    uint32_t need = static_cast<uint32_t>(k) - s_res[1];
    uint32_t cnt = s_res[2];

    // ---------------------------------------------------- further levels
    for (int l = 1; l < a.nlevels && cnt != need; ++l) {
        const int bl = a.bits[l];
        const int nsh = shift - bl;
        const int nb = 1 << bl;
        const uint32_t mask = static_cast<uint32_t>(nb - 1);
        if (list_ok) {
            for (int i = tid; i < L; i += NT) {
                const uint32_t kk = T::key(buf[list[i]]);
                if ((kk >> shift) == prefix) atomicAdd(&hist[(kk >> nsh) & mask], 1u);
            }
        } else {
            for (int base = warp * 32; base < nvt; base += NT) {
                const int v = base + lane;
                if (v < nvt) {
                    E el[V];
                    T::unpack(vbuf[v], el);
#pragma unroll
                    for (int t = 0; t < V; ++t) {
                        const uint32_t kk = T::key(el[t]);
                        if ((v * V + t < len) && ((kk >> shift) == prefix)) atomicAdd(&hist[(kk >> nsh) & mask], 1u);
                    }
                }
            }
        }
        __syncthreads();
        reduce_decide(nb, exact_threshold(need));
        prefix = (prefix << bl) | s_res[0];
        need -= s_res[1];
        cnt = s_res[2];
        shift = nsh;
    }
    const uint32_t P = prefix;
    const int S = shift;
    const uint32_t E_need = need;  // keys of class P still to take, in column order

    // --------------------------------------------- ordered write of the k
    int32_t *glist = GATHER ? reinterpret_cast<int32_t *>(smem + a.smem_glist_off) : nullptr;
    auto exchange_cta_totals = [&](uint32_t tg, uint32_t te) {
        // (selected before this CTA, threshold-class keys before this CTA) over the cluster, in rank order
        if constexpr (CLUSTER) {
            // every CTA stores its two counts into slot `rank` of every CTA of the cluster
            if (tid < static_cast<int>(csize)) {
                const uint32_t r = static_cast<uint32_t>(tid);
                dsmem_store(map_to_rank(smem_addr(&s_all_g[rank]), r), tg);
                dsmem_store(map_to_rank(smem_addr(&s_all_e[rank]), r), te);
            }
            cluster_sync();
        } else {
            __syncthreads();
        }
        if (tid == 0) {
            uint32_t eqb = 0, selb = 0;
            if constexpr (CLUSTER) {
                for (uint32_t r = 0; r < rank; ++r) {
                    const uint32_t g = s_all_g[r], e = s_all_e[r];
                    selb += g + take_from_ties(E_need, eqb, e);
                    eqb += e;
                }
            }
            s_cta_sel[0] = selb;
            s_cta_sel[1] = tg + take_from_ties(E_need, eqb, te);
            s_eq_before = eqb;
        }
        __syncthreads();
    };

    if (list_ok) {
        const int m = (L + NT - 1) / NT;
        const int i0 = min(L, tid * m), i1 = min(L, i0 + m);
        uint32_t g = 0, q = 0;
        for (int i = i0; i < i1; ++i) {
            const uint32_t c = T::key(buf[list[i]]) >> S;
            g += c > P;
            q += c == P;
        }
        uint32_t tg, tq;
        (void)block_exclusive_scan<NT>(g, s_warp, tg);
        const uint32_t qx = block_exclusive_scan<NT>(q, s_warp, tq);
        exchange_cta_totals(tg, tq);
        uint32_t r = s_eq_before + qx;
        const uint32_t sel = g + take_from_ties(E_need, r, q);
        uint32_t ts;
        uint32_t pos = s_cta_sel[0] + block_exclusive_scan<NT>(sel, s_warp, ts);
        const uint32_t cta_base = s_cta_sel[0];
        for (int i = i0; i < i1; ++i) {
            const int o = list[i];
            const E e = buf[o];
            const uint32_t c = T::key(e) >> S;
            bool take = c > P;
            if (c == P) take = (r++ < E_need);
            if (take) {
                const int64_t col = lo + o;
                store_idx(a, row, pos, col);
                if (a.want_values) store_val<E>(a, row, pos, e);
                if (GATHER && static_cast<int64_t>(pos) < a.n_gather) glist[pos - cta_base] = static_cast<int32_t>(col);
                ++pos;
            }
        }
    } else {
        // full-slice fallback (threshold bin too large for the list): warp-segment counts, then an
        // ordered write in which every warp walks its own contiguous segment
        const int seg = ((len + W - 1) / W + 32 * V - 1) / (32 * V) * (32 * V);
        const int w_lo = min(len, warp * seg);
        const int w_hi = min(len, w_lo + seg);
        uint32_t gt = 0, eq = 0;
        for (int o = w_lo + lane * V; o < w_hi; o += 32 * V) {
            E el[V];
            T::unpack(*reinterpret_cast<const uint4 *>(buf + o), el);
#pragma unroll
            for (int t = 0; t < V; ++t) {
                if (o + t < w_hi) {
                    const uint32_t c = T::key(el[t]) >> S;
                    gt += c > P;
                    eq += c == P;
                }
            }
        }
        gt = __reduce_add_sync(kFull, gt);
        eq = __reduce_add_sync(kFull, eq);
        if (lane == 0) {
            s_wgt[warp] = gt;
            s_weq[warp] = eq;
        }
        __syncthreads();
        uint32_t tg = 0, te = 0;
        for (int w = 0; w < W; ++w) {
            tg += s_wgt[w];
            te += s_weq[w];
        }
        exchange_cta_totals(tg, te);
        if (tid == 0) {
            uint32_t ws = s_cta_sel[0], we = s_eq_before;
            for (int w = 0; w < W; ++w) {
                s_wsel_base[w] = ws;
                s_weq_base[w] = we;
                ws += s_wgt[w] + take_from_ties(E_need, we, s_weq[w]);
                we += s_weq[w];
            }
        }
        __syncthreads();
        const uint32_t cta_base = s_cta_sel[0];
        uint32_t eq_run = s_weq_base[warp];
        uint32_t sel_run = s_wsel_base[warp];
        for (int base = w_lo; base < w_hi; base += 32 * V) {
            const int o = base + lane * V;
            const bool ok = o < w_hi;
            E el[V];
            T::unpack(ok ? *reinterpret_cast<const uint4 *>(buf + o) : make_uint4(0u, 0u, 0u, 0u), el);
            uint32_t gm = 0, qm = 0;
#pragma unroll
            for (int t = 0; t < V; ++t) {
                if (ok && o + t < w_hi) {
                    const uint32_t c = T::key(el[t]) >> S;
                    gm |= static_cast<uint32_t>(c > P) << t;
                    qm |= static_cast<uint32_t>(c == P) << t;
                }
            }
            if (!__any_sync(kFull, (gm | qm) != 0u)) continue;
            uint32_t tq;
            uint32_t r = eq_run + warp_exclusive_scan(static_cast<uint32_t>(__popc(qm)), lane, tq);
            uint32_t sm = gm;
#pragma unroll
            for (int t = 0; t < V; ++t) {
                if ((qm >> t) & 1u) {
                    if (r < E_need) sm |= 1u << t;
                    ++r;
                }
            }
            uint32_t ts;
            uint32_t pos = sel_run + warp_exclusive_scan(static_cast<uint32_t>(__popc(sm)), lane, ts);
#pragma unroll
            for (int t = 0; t < V; ++t) {
                if ((sm >> t) & 1u) {
                    const int64_t col = lo + o + t;
                    store_idx(a, row, pos, col);
                    if (a.want_values) store_val<E>(a, row, pos, el[t]);
                    if (GATHER && static_cast<int64_t>(pos) < a.n_gather)
                        glist[pos - cta_base] = static_cast<int32_t>(col);
                    ++pos;
                }
            }
            eq_run += tq;
            sel_run += ts;
        }
    }

    // ---------------------------------------------------- fused gather
    if (GATHER) {
        __syncthreads();
        const int64_t g0 = s_cta_sel[0];
        const int64_t g1 = min(g0 + static_cast<int64_t>(s_cta_sel[1]), a.n_gather);
        if (g0 < g1) gather_rows_of<NT>(a, row, g0, g1, glist, 0);
    }
    // no cluster barrier here: after the totals exchange no CTA touches another CTA's shared memory
}

// Raises the kernel's dynamic shared-memory limit (and allows clusters above 8) once per device;
// later calls that need no more than what was set skip the driver call.
template <typename E, int NT, bool C, bool G>
cudaError_t prepare_variant(int cluster, size_t smem)
{
    constexpr int kMaxDevices = 64;
    static int set_smem[kMaxDevices] = {};
    static bool set_cluster[kMaxDevices] = {};
    auto kern = topk_kernel<E, NT, C, G>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    if (!cacheable || set_smem[dev] < static_cast<int>(smem)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (cacheable) set_smem[dev] = static_cast<int>(smem);
    }
    if (C && cluster > 8 && (!cacheable || !set_cluster[dev])) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        if (cacheable) set_cluster[dev] = true;
    }
    return cudaSuccess;
}

template <typename E, int NT, bool C, bool G>
cudaError_t launch_variant(int cluster, size_t smem, const TopkArgs &a, cudaStream_t stream)
{
    auto kern = topk_kernel<E, NT, C, G>;
    cudaError_t e = prepare_variant<E, NT, C, G>(cluster, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.rows * (C ? cluster : 1)), 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (C) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename E, int NT, bool C, bool G>
int max_clusters_variant(int cluster, size_t smem)
{
    auto kern = topk_kernel<E, NT, C, G>;
    if (prepare_variant<E, NT, C, G>(cluster, smem) != cudaSuccess) return 0;
    if (!C) {
        int blocks = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, NT, smem) != cudaSuccess) return 0;
        return blocks * device_sm_count();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Dispatch over (dtype, threads, cluster?, gather?) to one of the 24 instantiations.
template <typename E, int NT>
cudaError_t launch_nt(bool gather, int cluster, size_t smem, const TopkArgs &a, cudaStream_t s)
{
    if (cluster > 1)
        return gather ? launch_variant<E, NT, true, true>(cluster, smem, a, s)
                      : launch_variant<E, NT, true, false>(cluster, smem, a, s);
    return gather ? launch_variant<E, NT, false, true>(1, smem, a, s) : launch_variant<E, NT, false, false>(1, smem, a, s);
}

template <typename E, int NT>
int occupancy_nt(bool gather, int cluster, size_t smem)
{
    if (cluster > 1)
        return gather ? max_clusters_variant<E, NT, true, true>(cluster, smem)
                      : max_clusters_variant<E, NT, true, false>(cluster, smem);
    return gather ? max_clusters_variant<E, NT, false, true>(1, smem) : max_clusters_variant<E, NT, false, false>(1, smem);
}

template <typename E>
cudaError_t launch_e(int threads, bool gather, int cluster, size_t smem, const TopkArgs &a, cudaStream_t s)
{
    switch (threads) {
    case 128: return launch_nt<E, 128>(gather, cluster, smem, a, s);
    case 256: return launch_nt<E, 256>(gather, cluster, smem, a, s);
    case 512: return launch_nt<E, 512>(gather, cluster, smem, a, s);
    default: return cudaErrorInvalidValue;
    }
}

template <typename E>
int occupancy_e(int threads, bool gather, int cluster, size_t smem)
{
    switch (threads) {
    case 128: return occupancy_nt<E, 128>(gather, cluster, smem);
    case 256: return occupancy_nt<E, 256>(gather, cluster, smem);
    case 512: return occupancy_nt<E, 512>(gather, cluster, smem);
    default: return 0;
    }
}

}  // namespace
}  // namespace sel
