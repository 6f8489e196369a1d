// topk.cu -- batched row-wise top-k by radix select, one row per CTA or per
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
    if (mbar_try_wait(bar, parity)) return;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitCycles) {
            set_err(err, kStatusTimeout);
            return;
        }
    }
}

// One shared atomicAdd per distinct digit per warp.  All 32 lanes must call.
__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t digit, bool valid, int lane)
{
    const unsigned peers = __match_any_sync(kFull, valid ? digit : 0xffffffffu);
    if (valid && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], (uint32_t)__popc(peers));
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

// Threshold digit of a histogram h[0, nb): the digit d with
//   sum_{e > d} h[e] < need <= sum_{e >= d} h[e].
// Result in out[0] = d, out[1] = sum_{e > d} h[e], out[2] = h[d].  All threads call.
__device__ void find_threshold(const uint32_t *h, int nb, uint32_t need, uint32_t *out, uint32_t *wsum)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = nb > kThreads ? nb / kThreads : 1;
    const int lo = tid * per;
    uint32_t s = 0;
    if (lo < nb)
        for (int i = 0; i < per; ++i) s += h[lo + i];
    uint32_t inc = s;  // becomes the sum over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(kFull, inc, o);
        if (lane + o < 32) inc += y;
    }
    if (lane == 0) wsum[warp] = inc;
    __syncthreads();
    uint32_t above = inc - s;
    for (int w = warp + 1; w < kWarps; ++w) above += wsum[w];
    if (lo < nb && above < need && above + s >= need) {
        uint32_t acc = above;
        for (int i = per - 1; i >= 0; --i) {
            const uint32_t c = h[lo + i];
            if (acc + c >= need) {
                out[0] = (uint32_t)(lo + i);
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
__device__ void gather_rows_of(const TopkArgs &a, int64_t row, int64_t j0, int64_t j1, const int32_t *glist,
                               int64_t n_short)
{
    const int vpr = static_cast<int>(a.d >> 3);  // 16-byte vectors per key row
    const int64_t bb = row / a.rows_per_batch;
    const uint16_t *kb = a.key + bb * a.key_batch_stride;
    uint4 *ob = reinterpret_cast<uint4 *>(a.gather_out + row * a.n_gather * a.d);
    const int total = static_cast<int>(j1 - j0) * vpr;
#pragma unroll 4
    for (int t = threadIdx.x; t < total; t += kThreads) {
        const int jj = t / vpr;
        const int v = t - jj * vpr;
        const int64_t j = j0 + jj;
        int64_t p = glist ? static_cast<int64_t>(glist[jj]) : (j < n_short ? j : 0);
        if (p < 0) p = 0;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (p < a.comp_len)
            val = __ldg(reinterpret_cast<const uint4 *>(kb + p * a.key_row_stride) + v);
        else if (v == 0)
            set_err(a.err_flag, kStatusInval);
        __stcs(ob + j * vpr + v, val);
    }
}

template <typename E, bool CLUSTER, bool GATHER>
__global__ void __launch_bounds__(kThreads, 2) topk_kernel(const TopkArgs a)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t s_bar[kMaxChunks];
    __shared__ uint32_t s_wsum[kWarps];
    __shared__ uint32_t s_wgt[kWarps], s_weq[kWarps];
    __shared__ uint32_t s_wsel_base[kWarps], s_weq_base[kWarps];
    __shared__ uint32_t s_thr[3];
    __shared__ uint32_t s_tot[2];       // this CTA's (greater, equal) counts; read by the cluster
    __shared__ uint32_t s_cta_sel[2];   // (selected before this CTA, selected by this CTA)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = CLUSTER ? cluster_rank() : 0u;
    const uint32_t csize = CLUSTER ? cluster_size() : 1u;
    const int64_t row = CLUSTER ? static_cast<int64_t>(cluster_id_x()) : static_cast<int64_t>(blockIdx.x);

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
        for (int j = j0 + tid; j < j1; j += kThreads) {
            store_idx(a, row, j, j < n ? j : -1);
            if (a.want_values) store_val<E>(a, row, j, j < n ? xrow[j] : static_cast<E>(T::kFill));
        }
        if (GATHER) {
            const int64_t g1 = min(static_cast<int64_t>(j1), a.n_gather);
            if (j0 < g1) gather_rows_of(a, row, j0, g1, nullptr, n);
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

    if (tid == 0) {
        for (int c = 0; c < nchunks; ++c) mbar_init(&s_bar[c], 1);
        fence_mbar_init();
    }
    for (int i = tid; i < a.hist_bins; i += kThreads) hist[i] = 0u;
    if (CLUSTER) {
        uint32_t *m = reinterpret_cast<uint32_t *>(smem + a.smem_merge_off);
        int words = 0;
        for (int l = 0; l < a.nlevels; ++l) words += 1 << a.bits[l];
        for (int i = tid; i < words; i += kThreads) m[i] = 0u;
    }
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
    if (CLUSTER) cluster_sync();  // all CTAs started and merge buffers zeroed before any remote access

    // ------------------------------- pass 1: top digit, while chunks land
    const int sh0 = T::KB - a.bits[0];
    bool has_nan = false;
    for (int c = 0; c < nchunks; ++c) {
        wait_phase(&s_bar[c], 0u, a.err_flag);
        const uint32_t cb = min(kChunkBytes, bulk - static_cast<uint32_t>(c) * kChunkBytes);
        const int nv = static_cast<int>(cb >> 4);
        const uint4 *vb = reinterpret_cast<const uint4 *>(smem + static_cast<size_t>(c) * kChunkBytes);
        for (int base = warp * 32; base < nv; base += kThreads) {
            const int v = base + lane;
            const bool ok = v < nv;
            const uint4 q = ok ? vb[v] : make_uint4(0u, 0u, 0u, 0u);
            E el[V];
            T::unpack(q, el);
#pragma unroll
            for (int t = 0; t < V; ++t) {
                has_nan |= ok && T::is_nan(el[t]);
                hist_add(hist, T::key(el[t]) >> sh0, ok, lane);
            }
        }
    }
    {
        const int tail0 = static_cast<int>(bulk / sizeof(E));
        if (tid < len - tail0) {  // < 16 bytes left over: plain loads
            const E e = xrow[lo + tail0 + tid];
            buf[tail0 + tid] = e;
            has_nan |= T::is_nan(e);
            atomicAdd(&hist[T::key(e) >> sh0], 1u);
        }
    }
    if (__syncthreads_or(has_nan) && tid == 0 && a.nan_flag) atomicOr(a.nan_flag, 1);

    // --------------------------------------------------- radix levels
    uint32_t prefix = 0;     // selection class: (key >> shift) == prefix
    int shift = T::KB;
    uint32_t need = static_cast<uint32_t>(k);
    uint32_t merge_off = a.smem_merge_off;
    const int nvt = (len + V - 1) / V;
    for (int l = 0; l < a.nlevels; ++l) {
        const int bl = a.bits[l];
        const int nsh = shift - bl;
        const int nb = 1 << bl;
        const uint32_t mask = static_cast<uint32_t>(nb - 1);
        if (l > 0) {
            const uint4 *vb = reinterpret_cast<const uint4 *>(buf);
            for (int base = warp * 32; base < nvt; base += kThreads) {
                const int v = base + lane;
                const bool ok = v < nvt;
                const uint4 q = ok ? vb[v] : make_uint4(0u, 0u, 0u, 0u);
                E el[V];
                T::unpack(q, el);
#pragma unroll
                for (int t = 0; t < V; ++t) {
                    const uint32_t kk = T::key(el[t]);
                    const bool m = ok && (v * V + t < len) && ((kk >> shift) == prefix);
                    hist_add(hist, (kk >> nsh) & mask, m, lane);
                }
            }
            __syncthreads();
        }
        if (CLUSTER) {
            uint32_t *mrg = reinterpret_cast<uint32_t *>(smem + merge_off);
            for (int i = tid; i < nb; i += kThreads) {
                const uint32_t c = hist[i];
                if (c) dsmem_add(map_to_rank(smem_addr(&mrg[i]), 0u), c);
            }
            cluster_sync();
            for (int i = tid; i < nb; i += kThreads) hist[i] = dsmem_load(map_to_rank(smem_addr(&mrg[i]), 0u));
            __syncthreads();
            merge_off += static_cast<uint32_t>(nb) * 4u;
        }
        find_threshold(hist, nb, need, s_thr, s_wsum);
        const uint32_t d = s_thr[0], above = s_thr[1], cnt = s_thr[2];
        prefix = (l == 0) ? d : ((prefix << bl) | d);
        need -= above;
        shift = nsh;
        for (int i = tid; i < nb; i += kThreads) hist[i] = 0u;
        __syncthreads();
        if (cnt == need) break;  // every key of the threshold bin is selected
    }
    const uint32_t P = prefix;
    const int S = shift;
    const uint32_t E_need = need;  // keys of class P still to take, in column order

    // ----------------------------------------------- count per warp segment
    const int seg = ((len + kWarps - 1) / kWarps + 32 * V - 1) / (32 * V) * (32 * V);
    const int w_lo = min(len, warp * seg);
    const int w_hi = min(len, w_lo + seg);
    {
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
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t tg = 0, te = 0;
        for (int w = 0; w < kWarps; ++w) {
            tg += s_wgt[w];
            te += s_weq[w];
        }
        s_tot[0] = tg;
        s_tot[1] = te;
    }
    if (CLUSTER)
        cluster_sync();
    else
        __syncthreads();
    if (tid == 0) {
        uint32_t eqb = 0, selb = 0;
        if constexpr (CLUSTER) {
            for (uint32_t q = 0; q < rank; ++q) {
                const uint32_t g = dsmem_load(map_to_rank(smem_addr(&s_tot[0]), q));
                const uint32_t e = dsmem_load(map_to_rank(smem_addr(&s_tot[1]), q));
                selb += g + take_from_ties(E_need, eqb, e);
                eqb += e;
            }
        }
        s_cta_sel[0] = selb;
        uint32_t ws = selb, we = eqb;
        for (int w = 0; w < kWarps; ++w) {
            s_wsel_base[w] = ws;
            s_weq_base[w] = we;
            ws += s_wgt[w] + take_from_ties(E_need, we, s_weq[w]);
            we += s_weq[w];
        }
        s_cta_sel[1] = ws - selb;
    }
    __syncthreads();

    // --------------------------------------------- ordered write of the k
    int32_t *glist = GATHER ? reinterpret_cast<int32_t *>(smem + a.smem_glist_off) : nullptr;
    {
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
                    if (GATHER && static_cast<int64_t>(pos) < a.n_gather) glist[pos - cta_base] = static_cast<int32_t>(col);
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
        if (g0 < g1) gather_rows_of(a, row, g0, g1, glist, 0);
    }
    if (CLUSTER) cluster_sync();  // keep this CTA's shared memory alive until the cluster is done with it
}

template <typename E, bool C, bool G>
cudaError_t launch_variant(int cluster, size_t smem, const TopkArgs &a, cudaStream_t stream)
{
    auto kern = topk_kernel<E, C, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (C && cluster > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.rows * (C ? cluster : 1)), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
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

template <typename E, bool C, bool G>
int max_clusters_variant(int cluster, size_t smem)
{
    auto kern = topk_kernel<E, C, G>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return 0;
    if (!C) {
        int blocks = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, kThreads, smem) != cudaSuccess) return 0;
        return blocks * device_sm_count();
    }
    if (cluster > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
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

}  // namespace

cudaError_t launch_topk(int dtype, bool gather, int cluster, size_t smem, const TopkArgs &a, cudaStream_t stream)
{
    const bool c = cluster > 1;
    if (dtype == 0) {
        if (c) return gather ? launch_variant<uint32_t, true, true>(cluster, smem, a, stream)
                             : launch_variant<uint32_t, true, false>(cluster, smem, a, stream);
        return gather ? launch_variant<uint32_t, false, true>(1, smem, a, stream)
                      : launch_variant<uint32_t, false, false>(1, smem, a, stream);
    }
    if (c) return gather ? launch_variant<uint16_t, true, true>(cluster, smem, a, stream)
                         : launch_variant<uint16_t, true, false>(cluster, smem, a, stream);
    return gather ? launch_variant<uint16_t, false, true>(1, smem, a, stream)
                  : launch_variant<uint16_t, false, false>(1, smem, a, stream);
}

int topk_max_active_clusters(int dtype, bool gather, int cluster, size_t smem)
{
    const bool c = cluster > 1;
    if (dtype == 0) {
        if (c) return gather ? max_clusters_variant<uint32_t, true, true>(cluster, smem)
                             : max_clusters_variant<uint32_t, true, false>(cluster, smem);
        return gather ? max_clusters_variant<uint32_t, false, true>(1, smem)
                      : max_clusters_variant<uint32_t, false, false>(1, smem);
    }
    if (c) return gather ? max_clusters_variant<uint16_t, true, true>(cluster, smem)
                         : max_clusters_variant<uint16_t, true, false>(cluster, smem);
    return gather ? max_clusters_variant<uint16_t, false, true>(1, smem)
                  : max_clusters_variant<uint16_t, false, false>(1, smem);
}

size_t topk_smem_limit()
{
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    // leave room for the kernel's static shared memory (barriers, per-warp counters)
    return optin > 1024 ? static_cast<size_t>(optin) - 1024 : 0;
}

int device_sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace sel
