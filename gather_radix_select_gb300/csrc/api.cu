// api.cu -- the C ABI (include/sel.h): argument checks, launch planning and
// dispatch.  Host code only; every step of the computation runs in the
// kernels of topk.cu and gather.cu.
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/sel.h"
#include "sel_internal.h"

namespace {

constexpr int kInAlign = 16;   // bulk copies stage input rows: 16-byte rows
constexpr int kOutAlign = 16;  // output rows start on 16 bytes
constexpr int64_t kSliceTargetBytes = 64 * 1024;
constexpr int64_t kSliceMinBytes = 8 * 1024;

int elem_bytes(int dtype) { return dtype == SEL_F32 ? 4 : 2; }
int idx_bytes(int idx_dtype) { return idx_dtype == SEL_I64 ? 8 : 4; }
bool aligned(const void *p, int a) { return (reinterpret_cast<uintptr_t>(p) % static_cast<uintptr_t>(a)) == 0; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

struct Plan {
    int cluster = 1;
    int threads = 256;
    size_t smem = 0;
    sel::TopkArgs layout{};  // slice, digit plan and shared-memory offsets
};

void digit_plan(int dtype, int64_t cols, sel::TopkArgs &a)
{
    const bool small = cols <= 4096;  // small rows: 256-bin histograms are cheaper to clear and scan
    if (dtype == SEL_F32) {
        if (small) {
            a.nlevels = 4;
            a.bits[0] = a.bits[1] = a.bits[2] = a.bits[3] = 8;
        } else {
            a.nlevels = 3;
            a.bits[0] = 11;
            a.bits[1] = 11;
            a.bits[2] = 10;
            a.bits[3] = 0;
        }
    } else {
        a.nlevels = 2;
        a.bits[0] = small ? 8 : 11;
        a.bits[1] = small ? 8 : 5;
        a.bits[2] = a.bits[3] = 0;
    }
    int mb = 0;
    for (int l = 0; l < a.nlevels; ++l) mb = a.bits[l] > mb ? a.bits[l] : mb;
    a.hist_bins = 1 << mb;
}

// Threads per selection CTA for a slice of `slice` elements.
int threads_for(int64_t slice)
{
    if (slice <= 4096) return 128;
    if (slice <= 16384) return 256;
    return 512;
}

// Shared-memory layout of one CTA for a given slice; returns total bytes.
size_t layout_for(int dtype, int cluster, int64_t slice, int k, bool gather, int64_t n_gather, sel::TopkArgs &a)
{
    const int64_t e = elem_bytes(dtype);
    a.slice = slice;
    size_t off = static_cast<size_t>(round_up(slice * e, 128));
    a.smem_buf_bytes = static_cast<uint32_t>(off);
    a.smem_hist_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(a.hist_bins) * 4;
    a.smem_mask_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(round_up(ceil_div(slice, 16 / e), 16));
    // candidate list (16-bit offsets): this CTA's share of k with room for the threshold bin; a CTA
    // whose candidates do not fit works on its whole staged slice instead
    const int64_t share = cluster > 1 ? 2 * ceil_div(k, cluster) : static_cast<int64_t>(k);
    const int64_t want = share + 2048;
    const int64_t cap = slice < want ? slice : want;
    a.list_cap = static_cast<int32_t>(cap);
    a.smem_list_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(round_up(cap * 2, 16));
    a.smem_glist_off = static_cast<uint32_t>(off);
    if (gather) off += static_cast<size_t>(round_up(n_gather * 4, 16));
    return off;
}

int cached_max_clusters(int dtype, int threads, bool gather, int cluster, size_t smem)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, size_t>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, dtype, threads, gather ? 1 : 0, cluster, smem);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const int n = sel::topk_max_active_clusters(dtype, threads, gather, cluster, smem);
    std::lock_guard<std::mutex> g(mu);
    cache[key] = n;
    return n;
}

// First-pass histogram flavour: SEL_HIST_AGG=1 selects warp-aggregated atomics
// (__match_any_sync), anything else plain shared atomics (the default).
int hist_agg()
{
    static const int v = [] {
        const char *e = std::getenv("SEL_HIST_AGG");
        return (e && e[0] == '1') ? 1 : 0;
    }();
    return v;
}

// Tries a cluster size: slice, threads, layout, and whether it can be scheduled.
bool try_cluster(int dtype, int64_t rows, int64_t cols, int k, bool gather, int64_t n_gather, int64_t cs,
                 size_t limit, Plan &p, bool &too_big)
{
    const int64_t e = elem_bytes(dtype);
    const int64_t slice = round_up(ceil_div(cols > 0 ? cols : 1, cs), 64);
    too_big = slice > sel::kMaxSlice || slice * e > static_cast<int64_t>(sel::kMaxChunks) * sel::kChunkBytes;
    if (too_big) return false;
    sel::TopkArgs a = p.layout;
    const size_t smem = layout_for(dtype, static_cast<int>(cs), slice, k, gather, n_gather, a);
    if (smem > limit) {
        too_big = true;
        return false;
    }
    if (rows * cs > 0x7fffffffLL) return false;
    const int threads = threads_for(slice);
    if (cached_max_clusters(dtype, threads, gather, static_cast<int>(cs), smem) <= 0) return false;
    p.cluster = static_cast<int>(cs);
    p.threads = threads;
    p.smem = smem;
    p.layout = a;
    return true;
}

// Chooses CTAs per row (cluster), the slice each CTA stages and the digit plan.
int make_plan(int dtype, int64_t rows, int64_t cols, int k, bool gather, int64_t n_gather, Plan &p)
{
    digit_plan(dtype, cols, p.layout);
    p.layout.agg = hist_agg();
    p.layout.sample_step = 8;
    p.layout.sample_min_cols = 8192;
    const size_t limit = sel::topk_smem_limit();
    const int sms = sel::device_sm_count();
    if (limit == 0 || sms == 0) return SEL_ECUDA;
    const int64_t e = elem_bytes(dtype);
    const int64_t row_bytes = (cols > 0 ? cols : 1) * e;
    int64_t want = ceil_div(row_bytes, kSliceTargetBytes);
    if (rows < 2 * sms) {
        // few rows: split them further so that every SM gets work
        const int64_t par = ceil_div(2 * sms, rows > 0 ? rows : 1);
        const int64_t cap = ceil_div(row_bytes, kSliceMinBytes);
        const int64_t extra = par < cap ? par : cap;
        if (extra > want) want = extra;
    }
    if (want > sel::kMaxCluster) want = sel::kMaxCluster;
    if (want < 1) want = 1;
    bool too_big = false;
    // smallest cluster >= want whose slice fits in shared memory and can be scheduled
    for (int64_t cs = want; cs <= sel::kMaxCluster; ++cs)
        if (try_cluster(dtype, rows, cols, k, gather, n_gather, cs, limit, p, too_big)) return SEL_OK;
    // a cluster that large could not be scheduled: try smaller ones that still fit
    for (int64_t cs = want - 1; cs >= 1; --cs) {
        if (try_cluster(dtype, rows, cols, k, gather, n_gather, cs, limit, p, too_big)) return SEL_OK;
        if (too_big) break;
    }
    return SEL_EUNSUPPORTED;
}

// make_plan behind a cache: the plan depends only on the device and the call's shape.
int cached_plan(int dtype, int64_t rows, int64_t cols, int k, bool gather, int64_t n_gather, Plan &p)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, int64_t, int64_t, int, int64_t>, Plan> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEL_ECUDA;
    const auto key = std::make_tuple(dev, dtype, rows, cols, k, gather ? n_gather : -1);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            p = it->second;
            return SEL_OK;
        }
    }
    const int st = make_plan(dtype, rows, cols, k, gather, n_gather, p);
    if (st != SEL_OK) return st;
    std::lock_guard<std::mutex> g(mu);
    if (cache.size() > 4096) cache.clear();
    cache[key] = p;
    return SEL_OK;
}

int check_topk_args(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride, int k, int idx_dtype,
                    int want_values, const void *out_idx, int64_t out_idx_stride, const void *out_val,
                    int64_t out_val_stride, bool idx_required)
{
    if (dtype != SEL_F32 && dtype != SEL_BF16) return SEL_EINVAL;
    if (idx_dtype != SEL_I32 && idx_dtype != SEL_I64) return SEL_EINVAL;
    if (k < 1 || k > SEL_MAX_K) return SEL_EINVAL;
    if (rows < 0 || cols < 0 || stride < cols) return SEL_EINVAL;
    if (rows == 0) return SEL_OK;
    if (cols > 0 && !x) return SEL_EINVAL;
    if (idx_required && !out_idx) return SEL_EINVAL;
    if (out_idx && out_idx_stride < k) return SEL_EINVAL;
    if (want_values && (!out_val || out_val_stride < k)) return SEL_EINVAL;
    if (x && (!aligned(x, kInAlign) || (stride * elem_bytes(dtype)) % kInAlign != 0)) return SEL_EALIGN;
    if (out_idx && (!aligned(out_idx, kOutAlign) || (out_idx_stride * idx_bytes(idx_dtype)) % kOutAlign != 0))
        return SEL_EALIGN;
    if (want_values && (!aligned(out_val, kOutAlign) || (out_val_stride * elem_bytes(dtype)) % kOutAlign != 0))
        return SEL_EALIGN;
    return SEL_OK;
}

int check_gather_key(const void *key, int64_t b, int64_t comp_len, int64_t d, int64_t key_batch_stride,
                     int64_t key_row_stride, int64_t rows, const void *out)
{
    if (b < 1 || comp_len < 0 || d < 1 || rows < 0 || rows % b != 0) return SEL_EINVAL;
    if (key_batch_stride < 0 || key_row_stride < d) return SEL_EINVAL;
    if (!key || !out) return SEL_EINVAL;
    if ((d * 2) % 16 != 0 || (key_row_stride * 2) % 16 != 0 || (key_batch_stride * 2) % 16 != 0) return SEL_EALIGN;
    if (!aligned(key, 16) || !aligned(out, 16)) return SEL_EALIGN;
    return SEL_OK;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? SEL_OK : SEL_ECUDA; }

}  // namespace

extern "C" {

int sel_stride_requirement(int *in_align_bytes, int *out_align_bytes)
{
    if (in_align_bytes) *in_align_bytes = kInAlign;
    if (out_align_bytes) *out_align_bytes = kOutAlign;
    return SEL_OK;
}

const char *sel_strerror(int status)
{
    switch (status) {
    case SEL_OK: return "ok";
    case SEL_EINVAL: return "invalid argument";
    case SEL_EALIGN: return "pointer or row stride not aligned (see sel_stride_requirement)";
    case SEL_EUNSUPPORTED: return "unsupported shape or type";
    case SEL_ECUDA: return "CUDA runtime error";
    case SEL_ETIMEOUT: return "a bounded device wait timed out";
    default: return "unknown status";
    }
}

int64_t sel_max_cols(int dtype)
{
    if (dtype != SEL_F32 && dtype != SEL_BF16) return 0;
    const size_t limit = sel::topk_smem_limit();
    if (limit == 0) return 0;
    // widest row: the largest schedulable cluster with the largest slice that fits in shared memory
    for (int64_t cs = sel::kMaxCluster; cs >= 1; --cs) {
        int64_t lo = 64, hi = sel::kMaxSlice;
        Plan best;
        bool found = false;
        while (lo <= hi) {  // largest slice (multiple of 64) that fits and schedules, at k = SEL_MAX_K
            const int64_t mid = (lo + hi) / 2 / 64 * 64;
            Plan p;
            digit_plan(dtype, mid * cs, p.layout);
            bool too_big = false;
            if (try_cluster(dtype, 1, mid * cs, SEL_MAX_K, false, 0, cs, limit, p, too_big) && p.cluster == cs) {
                best = p;
                found = true;
                lo = mid + 64;
            } else {
                hi = mid - 64;
            }
        }
        if (found) return best.layout.slice * cs;
    }
    return 0;
}

int sel_topk(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride, const int32_t *row_end, int k,
             int sorted_index, int idx_dtype, int want_values, void *out_idx, int64_t out_idx_stride, void *out_val,
             int64_t out_val_stride, int32_t *nan_flag, int32_t *err_flag, void *stream)
{
    (void)sorted_index;  // the ordered compaction always yields ascending column order
    int st = check_topk_args(x, dtype, rows, cols, stride, k, idx_dtype, want_values, out_idx, out_idx_stride, out_val,
                             out_val_stride, true);
    if (st != SEL_OK || rows == 0) return st;
    Plan p;
    st = cached_plan(dtype, rows, cols, k, false, 0, p);
    if (st != SEL_OK) return st;
    sel::TopkArgs a = p.layout;
    a.x = x;
    a.rows = rows;
    a.cols = cols;
    a.stride = stride;
    a.row_end = row_end;
    a.k = k;
    a.idx_i64 = idx_dtype == SEL_I64;
    a.want_values = want_values ? 1 : 0;
    a.out_idx = out_idx;
    a.out_idx_stride = out_idx_stride;
    a.out_val = want_values ? out_val : nullptr;
    a.out_val_stride = out_val_stride;
    a.nan_flag = nan_flag;
    a.err_flag = err_flag;
    a.rows_per_batch = 1;
    return status_of(sel::launch_topk(dtype == SEL_F32 ? 0 : 1, p.threads, false, p.cluster, p.smem, a,
                                      static_cast<cudaStream_t>(stream)));
}

int sel_gather_rows(const void *key, int64_t b, int64_t comp_len, int64_t d, int64_t key_batch_stride,
                    int64_t key_row_stride, const void *idx, int idx_dtype, int64_t rows, int64_t n,
                    int64_t idx_row_stride, void *out, int32_t *err_flag, void *stream)
{
    if (idx_dtype != SEL_I32 && idx_dtype != SEL_I64) return SEL_EINVAL;
    if (n < 0 || rows < 0) return SEL_EINVAL;
    if (rows == 0 || n == 0) return (b >= 1 && rows % (b > 0 ? b : 1) == 0) ? SEL_OK : SEL_EINVAL;
    int st = check_gather_key(key, b, comp_len, d, key_batch_stride, key_row_stride, rows, out);
    if (st != SEL_OK) return st;
    if (!idx || idx_row_stride < n) return SEL_EINVAL;
    sel::GatherArgs a{};
    a.key = static_cast<const uint16_t *>(key);
    a.comp_len = comp_len;
    a.d = d;
    a.key_batch_stride = key_batch_stride;
    a.key_row_stride = key_row_stride;
    a.idx = idx;
    a.idx_i64 = idx_dtype == SEL_I64;
    a.rows = rows;
    a.n = n;
    a.idx_row_stride = idx_row_stride;
    a.rows_per_batch = rows / b;
    a.out = static_cast<uint16_t *>(out);
    a.err_flag = err_flag;
    return status_of(sel::launch_gather(a, static_cast<cudaStream_t>(stream)));
}

int sel_topk_gather(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride, const int32_t *row_end,
                    int k, int sorted_index, int idx_dtype, int want_values, void *out_idx, int64_t out_idx_stride,
                    void *out_val, int64_t out_val_stride, const void *key, int64_t b, int64_t comp_len, int64_t d,
                    int64_t key_batch_stride, int64_t key_row_stride, int64_t n_gather, void *gather_out,
                    int32_t *nan_flag, int32_t *err_flag, void *stream)
{
    (void)sorted_index;
    int st = check_topk_args(x, dtype, rows, cols, stride, k, idx_dtype, want_values, out_idx, out_idx_stride, out_val,
                             out_val_stride, false);
    if (st != SEL_OK) return st;
    if (n_gather < 0 || n_gather > k) return SEL_EINVAL;
    if (rows == 0) return (b >= 1) ? SEL_OK : SEL_EINVAL;
    if (n_gather > 0) {
        st = check_gather_key(key, b, comp_len, d, key_batch_stride, key_row_stride, rows, gather_out);
        if (st != SEL_OK) return st;
    }
    Plan p;
    st = cached_plan(dtype, rows, cols, k, n_gather > 0, n_gather, p);
    if (st != SEL_OK) return st;
    sel::TopkArgs a = p.layout;
    a.x = x;
    a.rows = rows;
    a.cols = cols;
    a.stride = stride;
    a.row_end = row_end;
    a.k = k;
    a.idx_i64 = idx_dtype == SEL_I64;
    a.want_values = want_values ? 1 : 0;
    a.out_idx = out_idx;
    a.out_idx_stride = out_idx_stride;
    a.out_val = want_values ? out_val : nullptr;
    a.out_val_stride = out_val_stride;
    a.nan_flag = nan_flag;
    a.err_flag = err_flag;
    a.key = static_cast<const uint16_t *>(key);
    a.comp_len = comp_len;
    a.d = d;
    a.key_batch_stride = key_batch_stride;
    a.key_row_stride = key_row_stride;
    a.rows_per_batch = n_gather > 0 ? rows / b : 1;
    a.n_gather = n_gather;
    a.gather_out = static_cast<uint16_t *>(gather_out);
    return status_of(sel::launch_topk(dtype == SEL_F32 ? 0 : 1, p.threads, n_gather > 0, p.cluster, p.smem, a,
                                      static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
