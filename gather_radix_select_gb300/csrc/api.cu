// api.cu -- the C ABI (include/sel.h): argument checks, launch planning and
// dispatch.  Host code only; every step of the computation runs in the
// kernels of topk.cu and gather.cu.
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/sel.h"
#include "../../include/sel_tuning.h"
#include "order_core.cuh"
#include "sel_internal.h"

namespace {

constexpr int kInAlign = 16;   // bulk copies stage input rows: 16-byte rows
constexpr int kOutAlign = 16;  // output rows start on 16 bytes
constexpr int64_t kSliceTargetBytes = 32 * 1024;  // split_kernel: bytes of a row per CTA
constexpr int64_t kSliceMinBytes = 16 * 1024;     // ... at least, when splitting further for parallelism
constexpr int64_t kSplitMinRowBytes = 64 * 1024;  // rows narrower than this never split
constexpr int64_t kWideMaxRowBytes = 4 << 20;     // wider rows, when few, split over CTAs instead
constexpr int kWideHistBins = 2048;               // wide_kernel's range histogram (select_regions)
constexpr int64_t kRegMaxRowBytes = 16 * 1024;    // longer rows take the staged row kernel by default
constexpr int kWideSplitCtasPerSm = 6;            // wide rows: split them until this many CTAs per SM
constexpr int64_t kWidePartMinBytes = 32 * 1024;  // ... but no part smaller than this
constexpr int64_t kFlatChunkMaxVecs = 8192;       // flat_kernel: 128 KB chunks at most
constexpr int64_t kFlatChunkMinVecs = 256;        // ... and 4 KB at least

int elem_bytes(int dtype) { return dtype == SEL_F32 ? 4 : 2; }
int idx_bytes(int idx_dtype) { return idx_dtype == SEL_I64 ? 8 : 4; }
bool aligned(const void *p, int a) { return (reinterpret_cast<uintptr_t>(p) % static_cast<uintptr_t>(a)) == 0; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

struct Plan {
    int mode = sel::kModeRow;
    int threads = 256;
    int64_t grid = 0;
    size_t smem = 0;
    size_t ws_bytes = 0;
    sel::TopkArgs layout{};  // digit plan, slice, parts, shared-memory offsets, workspace layout
};

void digit_plan(int dtype, int64_t cols, sel::TopkArgs &a)
{
    const bool small = cols <= 4096;  // short bf16 rows: 256-bin histograms are cheaper to clear and scan
    if (dtype == SEL_F32) {
        a.nlevels = 3;
        a.bits[0] = 11;
        a.bits[1] = 11;
        a.bits[2] = 10;
        a.bits[3] = 0;
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

// Threads per row_kernel CTA for a row of `slice` elements.
int threads_for(int64_t slice)
{
    if (slice <= 4096) return 128;
    if (slice <= 16384) return 256;
    return 512;
}

// Shared-memory layout of one CTA staging `slice` elements with a candidate list of `cap`
// entries: slice | masks | list | histogram | gather list.  Everything in front of the histogram
// doubles as the staging area of split_kernel's merge.  Returns the total bytes.
size_t layout_staged(int dtype, int64_t slice, int64_t cap, bool gather, int64_t n_gather, sel::TopkArgs &a)
{
    const int64_t e = elem_bytes(dtype);
    a.slice = slice;
    size_t off = static_cast<size_t>(round_up(slice * e, 128));
    a.smem_buf_bytes = static_cast<uint32_t>(off);
    a.smem_mask_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(round_up(ceil_div(slice, 16 / e), 16));
    a.list_cap = static_cast<int32_t>(cap);
    a.smem_list_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(round_up(cap * 2, 16));
    a.smem_hist_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(a.hist_bins) * 4;
    a.smem_glist_off = static_cast<uint32_t>(off);
    if (gather) off += static_cast<size_t>(round_up(n_gather * 4, 16));
    return off;
}

// Layout of a reg_kernel CTA: histogram | source column per output position (16-bit) | gather
// list.  Returns the total bytes.
size_t layout_reg(int k, bool gather, int64_t n_gather, sel::TopkArgs &a)
{
    a.slice = 0;
    a.smem_buf_bytes = 0;
    a.smem_hist_off = 0;
    size_t off = static_cast<size_t>(a.hist_bins) * 4;
    a.smem_list_off = a.smem_mask_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(round_up(static_cast<int64_t>(k) * 2, 16));
    a.list_cap = 0;
    a.smem_glist_off = static_cast<uint32_t>(off);
    if (gather) off += static_cast<size_t>(round_up(n_gather * 4, 16));
    return off;
}

// Layout of a stream_kernel CTA (histogram and gather list only).
size_t layout_stream(bool gather, int64_t n_gather, sel::TopkArgs &a)
{
    a.slice = 0;
    a.smem_buf_bytes = 0;
    a.smem_hist_off = 0;
    size_t off = static_cast<size_t>(a.hist_bins) * 4;
    a.smem_mask_off = a.smem_list_off = static_cast<uint32_t>(off);
    a.list_cap = 0;
    a.smem_glist_off = static_cast<uint32_t>(off);
    if (gather) off += static_cast<size_t>(round_up(n_gather * 4, 16));
    return off;
}

// Workspace layout of split_kernel (see topk_impl.cuh); returns the total bytes.
size_t layout_workspace(int dtype, int64_t rows, int parts, int64_t cap, sel::TopkArgs &a)
{
    a.parts = parts;
    a.ws_counter_bytes = round_up(rows * 4, 256);
    a.ws_head_bytes = round_up(2 * static_cast<int64_t>(parts) * 4, 16);
    a.ws_bits_bytes = round_up(cap * elem_bytes(dtype), 16);
    a.ws_part_bytes = a.ws_bits_bytes + round_up(cap * 4, 16);
    a.ws_row_bytes = a.ws_head_bytes + static_cast<int64_t>(parts) * a.ws_part_bytes;
    return static_cast<size_t>(a.ws_counter_bytes + rows * a.ws_row_bytes);
}

// Tuning knobs (include/sel_tuning.h): read from the environment once, when first needed, and
// settable at any time through sel_set_tuning.  The plan cache is keyed on them.
struct Tuning {
    std::atomic<int> plan{SEL_PLAN_AUTO}, parts{0}, row_sample{0}, hist_agg{0}, row_order{0};
};

int plan_from_name(const char *v)
{
    if (!v) return SEL_PLAN_AUTO;
    if (!std::strcmp(v, "reg")) return SEL_PLAN_REG;
    if (!std::strcmp(v, "row")) return SEL_PLAN_ROW;
    if (!std::strcmp(v, "wide")) return SEL_PLAN_WIDE;
    if (!std::strcmp(v, "split")) return SEL_PLAN_SPLIT;
    if (!std::strcmp(v, "stream")) return SEL_PLAN_STREAM;
    if (!std::strcmp(v, "flat")) return SEL_PLAN_FLAT;
    return SEL_PLAN_AUTO;
}

Tuning &tuning()
{
    static Tuning *t = [] {
        Tuning *n = new Tuning();
        n->plan = plan_from_name(std::getenv("SEL_PLAN"));
        const char *e = std::getenv("SEL_PARTS");
        const int v = e ? std::atoi(e) : 0;
        n->parts = v > 0 ? v : 0;
        e = std::getenv("SEL_ROW_SAMPLE");
        n->row_sample = (e && e[0] == '1') ? 1 : 0;
        e = std::getenv("SEL_HIST_AGG");
        n->hist_agg = (e && e[0] == '1') ? 1 : 0;
        e = std::getenv("SEL_ROW_ORDER");
        n->row_order = (e && e[0] == '1') ? 1 : 0;
        return n;
    }();
    return *t;
}

// SEL_PLAN_* -> the kernel mode it forces (-1: none)
int forced_mode(int plan)
{
    switch (plan) {
    case SEL_PLAN_REG: return sel::kModeReg8;
    case SEL_PLAN_ROW: return sel::kModeRow;
    case SEL_PLAN_WIDE: return sel::kModeWide;
    case SEL_PLAN_SPLIT: return sel::kModeSplit;
    case SEL_PLAN_STREAM: return sel::kModeStream;
    case SEL_PLAN_FLAT: return sel::kModeFlat;
    default: return -1;
    }
}

int cached_blocks_per_sm(int dtype, int mode, int threads, bool gather, size_t smem)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int, size_t>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, dtype, mode, threads, gather ? 1 : 0, smem);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const int n = sel::topk_blocks_per_sm(dtype, mode, threads, gather, smem);
    std::lock_guard<std::mutex> g(mu);
    cache[key] = n;
    return n;
}

// Candidate capacity of wide_kernel for rows of `cols` elements.  The threshold is estimated
// from a sample of up to kWideThreads * kWideSampleVecsPerLane 16-byte vectors (mu = k * sample / cols of the k
// expected there, keeping mu * 9/8 + 3 sqrt(mu) + 4 sampled keys); the list holds that many
// scaled to the row, plus four standard deviations of the count.
int64_t wide_cap(int dtype, int64_t cols, int k)
{
    const int64_t e = elem_bytes(dtype);
    const int64_t nvec = cols * e / 16;
    const int64_t sample =
        std::min<int64_t>(nvec, static_cast<int64_t>(sel::kWideThreads) * sel::kWideSampleVecsPerLane) * (16 / e);
    if (sample <= 0) return round_up(cols, 8);
    const double f = static_cast<double>(sample) / static_cast<double>(cols);
    const double mu = static_cast<double>(k) * f;
    const double kept = mu * 1.125 + 3.0 * std::sqrt(mu) + 4.0;
    const int64_t cap = static_cast<int64_t>((kept + 4.0 * std::sqrt(kept)) / f) + 64;
    return std::min(cap, round_up(cols, 8));
}

// Candidate pairs one of P parts of a row may leave (its part of wide_cap: the part estimates the
// row's threshold from its own sample, so it keeps its share of what the whole row would keep).
int64_t wide_part_cap(int dtype, int64_t cols, int k, int parts)
{
    const int64_t e = elem_bytes(dtype);
    const int64_t part_cols = ceil_div(cols, parts);
    const int64_t nvec = part_cols * e / 16;
    const int64_t sample =
        std::min<int64_t>(nvec, static_cast<int64_t>(sel::kWideThreads) * sel::kWideSampleVecsPerLane) * (16 / e);
    if (sample <= 0) return round_up(part_cols, 8);
    const double f = static_cast<double>(sample) / static_cast<double>(part_cols);
    const double mu = static_cast<double>(k) * static_cast<double>(sample) / static_cast<double>(cols);
    const double kept = mu * 1.125 + 3.0 * std::sqrt(mu) + 4.0;
    const int64_t cap = static_cast<int64_t>((kept + 4.0 * std::sqrt(kept)) / f) + 64;
    return std::min(cap, round_up(part_cols, 8) + 8);
}

// Layout of a wide_kernel CTA: histogram | W candidate regions of (key bits, column) pairs |
// gather list.  Each warp's region holds its share of `cap` plus slack for the uneven spread
// of candidates over the warps, and one more pair that absorbs writes past the capacity.
size_t layout_wide(int64_t cap, bool gather, int64_t n_gather, sel::TopkArgs &a)
{
    constexpr int W = sel::kWideThreads / 32;
    const int64_t per = ceil_div(cap, W);
    const int64_t capw = per + static_cast<int64_t>(4.0 * std::sqrt(static_cast<double>(per))) + 16;
    a.slice = 0;
    a.smem_buf_bytes = 0;
    a.smem_hist_off = 0;
    a.hist_bins = std::max(a.hist_bins, kWideHistBins);  // also holds the range histogram
    size_t off = static_cast<size_t>(a.hist_bins) * 4;
    a.list_cap = static_cast<int32_t>(capw);
    a.region_stride = static_cast<int32_t>(round_up(capw + 1, 2));
    a.smem_list_off = static_cast<uint32_t>(off);
    a.smem_mask_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(W) * static_cast<size_t>(a.region_stride) * 8;
    a.smem_glist_off = static_cast<uint32_t>(off);
    if (gather) off += static_cast<size_t>(round_up(n_gather * 4, 16));
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off), 16));
    a.smem_stage_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(W) * sel::kWideStage * (16 + 4);
    return off;
}

// Layout of a flat_kernel launch (topk_impl.cuh): each row's full 16-byte vectors cut into
// `parts` chunks of `slice` vectors, chunk q on CTA q mod grid (one CTA per SM).  Capacities
// follow the threshold estimate's margins: the estimate keeps about kept = mu*9/8 + 3 sqrt(mu) + 4
// of the m sampled keys (mu = k * m / cols), so a share e of the row holds about e * kept / m
// candidates; four standard deviations are added on top.
bool plan_flat(int dtype, int64_t rows, int64_t cols, int k, int sms, size_t limit, Plan &fp)
{
    sel::TopkArgs &a = fp.layout;
    constexpr int SW = sel::kFlatStreamWarps;
    const int64_t e = elem_bytes(dtype);
    const int64_t V = 16 / e;
    const int64_t nvr = cols * e / 16;
    if (nvr < 1 || sms < 1 || cols > 0x7fffffffLL) return false;
    int64_t cv = std::min(kFlatChunkMaxVecs, std::max(kFlatChunkMinVecs, ceil_div(rows * nvr, sms)));
    cv = std::max(cv, ceil_div(nvr, sel::kFlatMaxParts));  // chunks of a row bounded
    const int64_t cpr = ceil_div(nvr, cv);
    cv = ceil_div(nvr, cpr);
    if (cpr > sel::kFlatMaxParts || ceil_div(rows * cpr, sms) > sel::kFlatQueue) return false;
    const double m = static_cast<double>(std::min<int64_t>(nvr, sel::kFlatSampleVecs) * V);
    const double mu = static_cast<double>(k) * m / static_cast<double>(cols);
    const double kept = mu * 1.125 + 3.0 * std::sqrt(mu) + 4.0;
    const double frac = std::min(1.0, (kept + 4.0 * std::sqrt(kept)) / m);
    const double ew = static_cast<double>(ceil_div(cv, SW) * V);  // one streaming warp's share of a chunk
    const int64_t wcap = std::min<int64_t>(static_cast<int64_t>(ew) + 2 * V,
                                           static_cast<int64_t>(ew * frac + 4.0 * std::sqrt(ew * frac) + 16.0) + V);
    const double cf = static_cast<double>(cols) * frac;
    const int64_t total_cap = std::min<int64_t>(round_up(cols, 8), static_cast<int64_t>(cf + 4.0 * std::sqrt(cf)) + 64);
    const int64_t rs8 = round_up(ceil_div(total_cap, sel::kFlatSelWarps) + 17, 2);  // a region and its spare pair
    a.hist_bins = std::max(a.hist_bins, kWideHistBins);
    a.slice = cv;
    a.parts = static_cast<int32_t>(cpr);
    a.flat_wcap = static_cast<int32_t>(wcap);
    a.part_cap = static_cast<int32_t>(SW * wcap);  // a chunk's slot: every warp's region, concatenated
    a.flat_sel_pairs = static_cast<int32_t>(sel::kFlatSelWarps * rs8);
    a.list_cap = 0;
    a.region_stride = 0;
    a.smem_buf_bytes = 0;
    a.smem_mask_off = 0;
    a.smem_hist_off = 0;
    size_t off = static_cast<size_t>(a.hist_bins) * 4;
    a.smem_list_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(a.flat_sel_pairs) * 8;
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off), 16));
    a.smem_glist_off = static_cast<uint32_t>(off);
    a.smem_stage_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(SW) * sel::kWideStage * (16 + 4);
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off), 16));
    a.smem_cbuf_off = static_cast<uint32_t>(off);
    off += static_cast<size_t>(sel::kFlatBufs) * SW * static_cast<size_t>(wcap + 1) * 8;
    if (off > limit || cached_blocks_per_sm(dtype, sel::kModeFlat, sel::kFlatThreads, false, off) < 1) return false;
    a.ws_counter_bytes = round_up(3 * rows * 4, 256);
    a.ws_part_bytes = round_up(16 + SW * wcap * 8, 16);
    a.ws_row_bytes = cpr * a.ws_part_bytes;
    fp.mode = sel::kModeFlat;
    fp.threads = sel::kFlatThreads;
    fp.smem = off;
    fp.grid = sms;
    fp.ws_bytes = static_cast<size_t>(a.ws_counter_bytes + rows * a.ws_row_bytes);
    return true;
}

// Chooses the kernel (row / split / wide / stream), its CTA shape, shared memory and workspace.
int make_plan(int dtype, int64_t rows, int64_t cols, int k, bool gather, int64_t n_gather, int force, int force_parts,
              Plan &p)
{
    sel::TopkArgs &a = p.layout;
    digit_plan(dtype, cols, a);
    a.agg = tuning().hist_agg.load(std::memory_order_relaxed);
    a.sample_step = tuning().row_sample.load(std::memory_order_relaxed) ? 8 : 1;
    a.sample_min_cols = 8192;
    const size_t limit = sel::topk_smem_limit();
    const int sms = sel::device_sm_count();
    if (limit == 0 || sms == 0) return SEL_ECUDA;
    const int64_t e = elem_bytes(dtype);
    const int64_t c1 = cols > 0 ? cols : 1;
    const int64_t row_bytes = c1 * e;
    const int64_t max_staged = std::min<int64_t>(sel::kMaxSlice, sel::kMaxChunks * sel::kChunkBytes / e);

    // one CTA per row held in registers: the smallest tile (threads x 16-byte vectors a thread)
    // that holds the row
    bool reg_ok = false;
    Plan reg_plan = p;
    {
        struct Tile {
            int mode, threads, vecs;
        };
        const Tile tiles[] = {{sel::kModeReg2, 128, 2}, {sel::kModeReg8, 128, 8}, {sel::kModeReg8, 256, 8},
                              {sel::kModeReg8, 512, 8}};
        for (const Tile &t : tiles) {
            if (c1 > static_cast<int64_t>(t.threads) * t.vecs * (16 / e)) continue;
            Plan rp = p;
            const size_t smem = layout_reg(k, gather, n_gather, rp.layout);
            if (smem > limit || cached_blocks_per_sm(dtype, t.mode, t.threads, gather, smem) <= 0) continue;
            rp.mode = t.mode;
            rp.threads = t.threads;
            rp.smem = smem;
            rp.grid = rows;
            rp.ws_bytes = 0;
            reg_plan = rp;
            reg_ok = true;
            break;
        }
    }
    // measured: the register tiles beat the staged row kernel on rows of up to 1024 16-byte
    // vectors; on longer rows every radix pass over all registers costs more than the staged
    // kernel's sampled estimate and candidate list
    if (reg_ok && ((force < 0 && row_bytes <= kRegMaxRowBytes) || force == sel::kModeReg8)) {
        p = reg_plan;
        return SEL_OK;
    }
    // one CTA per row, the row staged whole
    bool row_ok = false;
    Plan row_plan = p;
    {
        const int64_t slice = round_up(c1, 64);
        if (slice <= max_staged) {
            const int64_t cap = std::min<int64_t>(slice, static_cast<int64_t>(k) + 2048);
            const size_t smem = layout_staged(dtype, slice, cap, gather, n_gather, row_plan.layout);
            const int threads = threads_for(slice);
            if (smem <= limit && cached_blocks_per_sm(dtype, sel::kModeRow, threads, gather, smem) > 0) {
                row_plan.mode = sel::kModeRow;
                row_plan.threads = threads;
                row_plan.smem = smem;
                row_plan.grid = rows;
                row_plan.ws_bytes = 0;
                row_ok = true;
            }
        }
    }
    // one CTA per row, one streaming pass into per-warp candidate lists; when the rows are fewer
    // than half the SMs, each row is streamed by `parts` CTAs whose candidate lists meet in the
    // workspace.  (Measured: a part carries ~10 us of fixed latency -- estimate, fences, merge --
    // so splitting pays only when most SMs would otherwise idle.)
    bool wide_ok = false;
    Plan wide_plan = p;
    if (cols <= 0x7fffffffLL) {
        int64_t parts = 1;
        if (2 * rows < sms) {
            parts = ceil_div(static_cast<int64_t>(kWideSplitCtasPerSm) * sms, rows > 0 ? rows : 1);
            parts = std::min<int64_t>(parts, std::max<int64_t>(1, row_bytes / kWidePartMinBytes));
            parts = std::min<int64_t>(parts, sel::kMaxParts);
        }
        if (force_parts > 0) parts = std::min<int64_t>(force_parts, sel::kMaxParts);
        Plan wp = p;
        const int64_t part_cap = parts > 1 ? wide_part_cap(dtype, c1, k, static_cast<int>(parts)) : 0;
        const int64_t cap = parts > 1 ? parts * part_cap : wide_cap(dtype, c1, k);
        const size_t smem = layout_wide(cap, gather, n_gather, wp.layout);
        const int mode = parts > 1 ? sel::kModeWideSplit : sel::kModeWide;
        if (smem <= limit && cached_blocks_per_sm(dtype, mode, sel::kWideThreads, gather, smem) > 0 &&
            rows * parts <= 0x7fffffffLL) {
            wp.mode = mode;
            wp.threads = sel::kWideThreads;
            wp.smem = smem;
            wp.grid = rows * parts;
            wp.ws_bytes = 0;
            if (parts > 1) {
                sel::TopkArgs &l = wp.layout;
                l.parts = static_cast<int32_t>(parts);
                l.part_cap = static_cast<int32_t>(part_cap);
                l.ws_counter_bytes = round_up(rows * 4, 256);
                l.ws_part_bytes = round_up(16 + part_cap * 8, 16);
                l.ws_row_bytes = parts * l.ws_part_bytes;
                wp.ws_bytes = static_cast<size_t>(l.ws_counter_bytes + rows * l.ws_row_bytes);
            }
            wide_plan = wp;
            wide_ok = true;
        }
    }
    if (force == sel::kModeRow && row_ok) {
        p = row_plan;
        return SEL_OK;
    }
    if (force == sel::kModeWide && wide_ok) {
        p = wide_plan;
        return SEL_OK;
    }
    // rows cut into chunks dealt over a persistent grid (flat_kernel): forced only, for now
    if (force == sel::kModeFlat) {
        Plan fp = p;
        if (!gather && plan_flat(dtype, rows, c1, k, sms, limit, fp)) {
            p = fp;
            return SEL_OK;
        }
    }
    // few wide rows (or rows that do not fit one CTA) leave the row plan
    const bool leave_row = !row_ok || (rows < 2 * sms && row_bytes >= kSplitMinRowBytes);
    if (!leave_row && force < 0) {
        p = row_plan;
        return SEL_OK;
    }
    if (force < 0 && wide_ok && !row_ok && (row_bytes <= kWideMaxRowBytes || rows >= sms)) {
        p = wide_plan;
        return SEL_OK;
    }
    if (force < 0 || force == sel::kModeSplit) {
        int64_t parts = ceil_div(row_bytes, kSliceTargetBytes);
        if (rows < 2 * sms) {
            const int64_t par = ceil_div(2 * sms, rows > 0 ? rows : 1);
            parts = std::max(parts, std::min(par, ceil_div(row_bytes, kSliceMinBytes)));
        }
        parts = std::max<int64_t>(2, std::min<int64_t>(parts, sel::kMaxParts));
        const int64_t slice = round_up(ceil_div(c1, parts), 64);
        parts = ceil_div(c1, slice);
        if (slice <= max_staged && parts >= 2) {
            Plan sp = p;
            const int64_t cap = std::min<int64_t>(slice, 2 * ceil_div(k, parts) + 512);
            const size_t smem = layout_staged(dtype, slice, cap, gather, n_gather, sp.layout);
            if (smem <= limit && cached_blocks_per_sm(dtype, sel::kModeSplit, 256, gather, smem) > 0 &&
                rows * parts <= 0x7fffffffLL) {
                sp.layout.sample_step = 4;  // each slice estimates its own threshold: a denser sample
                sp.mode = sel::kModeSplit;
                sp.threads = 256;
                sp.smem = smem;
                sp.grid = rows * parts;
                sp.ws_bytes = layout_workspace(dtype, rows, static_cast<int>(parts), cap, sp.layout);
                p = sp;
                return SEL_OK;
            }
        }
    }
    if (row_ok && force != sel::kModeStream) {
        p = row_plan;
        return SEL_OK;
    }
    if (wide_ok && force != sel::kModeStream) {
        p = wide_plan;
        return SEL_OK;
    }
    // otherwise one CTA per row, passes over global memory
    if (cols > 0x7fffffffLL) return SEL_EUNSUPPORTED;
    Plan st = p;
    const size_t smem = layout_stream(gather, n_gather, st.layout);
    if (smem > limit || cached_blocks_per_sm(dtype, sel::kModeStream, 512, gather, smem) <= 0) return SEL_EUNSUPPORTED;
    st.mode = sel::kModeStream;
    st.threads = 512;
    st.smem = smem;
    st.grid = rows;
    st.ws_bytes = 0;
    p = st;
    return SEL_OK;
}

// make_plan behind a cache: the plan depends only on the device, the call's shape and the tuning
// knobs.  A thread's last plan is kept in a thread-local entry, so repeated calls of one shape
// take no lock.
int cached_plan(int dtype, int64_t rows, int64_t cols, int k, bool gather, int64_t n_gather, Plan &p)
{
    using Key = std::tuple<int, int, int64_t, int64_t, int, int64_t, int, int, int>;
    static std::mutex mu;
    static std::map<Key, Plan> cache;
    thread_local bool last_valid = false;
    thread_local Key last_key;
    thread_local Plan last_plan;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEL_ECUDA;
    Tuning &t = tuning();
    const int force = forced_mode(t.plan.load(std::memory_order_relaxed));
    const int force_parts = t.parts.load(std::memory_order_relaxed);
    const int flavour = t.hist_agg.load(std::memory_order_relaxed) + 2 * t.row_sample.load(std::memory_order_relaxed);
    const Key key = std::make_tuple(dev, dtype, rows, cols, k, gather ? n_gather : -1, force, flavour, force_parts);
    if (last_valid && key == last_key) {
        p = last_plan;
        return SEL_OK;
    }
    bool found = false;
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            p = it->second;
            found = true;
        }
    }
    if (!found) {
        const int st = make_plan(dtype, rows, cols, k, gather, n_gather, force, force_parts, p);
        if (st != SEL_OK) return st;
        std::lock_guard<std::mutex> g(mu);
        if (cache.size() > 4096) cache.clear();
        cache[key] = p;
    }
    last_key = key;
    last_plan = p;
    last_valid = true;
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

// Elements from key[0] to the end of the key's last row (b batches of comp_len rows of d).
int64_t key_span(int64_t b, int64_t comp_len, int64_t d, int64_t batch_stride, int64_t row_stride)
{
    return comp_len > 0 && b > 0 ? (b - 1) * batch_stride + (comp_len - 1) * row_stride + d : 0;
}

// The key rows to gather after ordering (n_gather 0: none).
struct OrderGather {
    const void *key = nullptr;
    int64_t b = 1, comp_len = 0, d = 0, key_batch_stride = 0, key_row_stride = 0, n_gather = 0;
    void *gather_out = nullptr;
    int32_t *err_flag = nullptr;
};

// Re-orders finished output rows by value (SEL_SORT_VALUE), then gathers the first n_gather
// ordered positions' key rows in the same launch.
int value_order(const void *x, int dtype, int64_t rows, int64_t stride, int k, int idx_dtype, int want_values,
                void *out_idx, int64_t out_idx_stride, void *out_val, int64_t out_val_stride, void *stream,
                const OrderGather &g = OrderGather())
{
    sel::OrderArgs a{};
    if (g.n_gather > 0) {
        a.key = static_cast<const uint16_t *>(g.key);
        a.comp_len = g.comp_len;
        a.d = g.d;
        a.key_batch_stride = g.key_batch_stride;
        a.key_row_stride = g.key_row_stride;
        a.rows_per_batch = rows / g.b;
        a.key_span = key_span(g.b, g.comp_len, g.d, g.key_batch_stride, g.key_row_stride);
        a.n_gather = g.n_gather;
        a.gather_out = static_cast<uint16_t *>(g.gather_out);
        a.err_flag = g.err_flag;
    }
    a.x = x;
    a.x_stride = stride;
    a.rows = rows;
    a.k = k;
    a.out_idx = out_idx;
    a.out_idx_stride = out_idx_stride;
    a.out_val = want_values ? out_val : nullptr;
    a.out_val_stride = out_val_stride;
    return status_of(sel::launch_value_order(dtype, idx_dtype == SEL_I64, a, static_cast<cudaStream_t>(stream)));
}

// The value-ordered variant of a plan, where the selection kernel ranks its own outputs: the
// staged row kernel, whose ranking takes the (then free) masks and candidate list and, where those
// are too small, pushes the histogram and gather list back; or, for calls with a fused gather, the
// register kernel, whose ranking goes after its histogram, position table and gather list.  k must
// fit 8 entries a thread, and for the row kernel the 16-bit position slots of the histogram.  False
// for every other plan, or when the ranking does not fit.
bool ordered_plan(int dtype, int k, bool gather, const Plan &p, Plan &op)
{
    if (k > sel::order::kEpt * p.threads || k > (1 << sel::order::kSlotBits)) return false;
    const size_t rank = dtype == SEL_BF16 ? sel::order::rank_smem_bytes<true>(p.threads)
                                          : sel::order::rank_smem_bytes<false>(p.threads);
    op = p;
    sel::TopkArgs &l = op.layout;
    if (p.mode == sel::kModeRow) {
        if (k > 2 * p.layout.hist_bins) return false;
        l.smem_order_off = l.smem_mask_off;
        const size_t hist = static_cast<size_t>(
            round_up(static_cast<int64_t>(std::max<size_t>(l.smem_hist_off, l.smem_order_off + rank)), 16));
        const size_t delta = hist - l.smem_hist_off;
        l.smem_hist_off = static_cast<uint32_t>(hist);
        l.smem_glist_off = static_cast<uint32_t>(l.smem_glist_off + delta);
        op.smem = p.smem + delta;
        op.mode = sel::kModeRowOrdered;
    } else if ((p.mode == sel::kModeReg2 || p.mode == sel::kModeReg8) && gather) {
        // measured: with a fused gather, ranking in the register kernel saves the ordering launch's
        // index round trip (bf16 [4096, 2048] causal k=512 + gather 512: 0.119 -> 0.103 ms); without
        // one, the ordering launch ranks with more parallelism than the selection's epilogue
        // (0.050 against 0.052-0.054 ms), so it keeps the second launch
        l.smem_order_off = static_cast<uint32_t>(round_up(static_cast<int64_t>(p.smem), 16));
        op.smem = l.smem_order_off + rank;
        op.mode = p.mode == sel::kModeReg2 ? sel::kModeReg2Ordered : sel::kModeReg8Ordered;
    } else {
        return false;
    }
    return op.smem <= sel::topk_smem_limit() && cached_blocks_per_sm(dtype, op.mode, op.threads, gather, op.smem) > 0;
}

// One selection launch.  ordered (nullable): on entry, whether the outputs should come out in value
// order from this launch; when the plan cannot, nothing is launched and *ordered becomes false.
int run_topk(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride, const int32_t *row_end, int k,
             int idx_dtype, int want_values, void *out_idx, int64_t out_idx_stride, void *out_val,
             int64_t out_val_stride, const void *key, int64_t b, int64_t comp_len, int64_t d,
             int64_t key_batch_stride, int64_t key_row_stride, int64_t n_gather, void *gather_out, void *workspace,
             size_t workspace_bytes, int32_t *nan_flag, int32_t *err_flag, void *stream, int64_t row_end_div = 1,
             bool *ordered = nullptr)
{
    Plan p;
    int st = cached_plan(dtype, rows, cols, k, n_gather > 0, n_gather, p);
    if (st != SEL_OK) return st;
    if (ordered && *ordered) {
        Plan op;
        if (!ordered_plan(dtype, k, n_gather > 0, p, op)) {
            *ordered = false;
            return SEL_OK;
        }
        p = op;
    }
    if (p.ws_bytes > 0) {
        if (!workspace || workspace_bytes < p.ws_bytes) return SEL_EINVAL;
        if (!aligned(workspace, 256)) return SEL_EALIGN;
    }
    sel::TopkArgs a = p.layout;
    a.x = x;
    a.rows = rows;
    a.cols = cols;
    a.stride = stride;
    a.row_end = row_end;
    a.row_end_div = row_end_div;
    a.row_order = row_end && tuning().row_order.load(std::memory_order_relaxed) ? 1 : 0;
    a.k = k;
    a.idx_i64 = idx_dtype == SEL_I64;
    a.want_values = want_values ? 1 : 0;
    a.out_idx = out_idx;
    a.out_idx_stride = out_idx_stride;
    a.out_val = want_values ? out_val : nullptr;
    a.out_val_stride = out_val_stride;
    a.nan_flag = nan_flag;
    a.err_flag = err_flag;
    a.ws = static_cast<unsigned char *>(workspace);
    a.ws_bytes = workspace ? workspace_bytes : 0;
    a.key = static_cast<const uint16_t *>(key);
    a.comp_len = comp_len;
    a.d = d;
    a.key_batch_stride = key_batch_stride;
    a.key_row_stride = key_row_stride;
    a.rows_per_batch = n_gather > 0 ? rows / b : 1;
    a.key_span = n_gather > 0 ? key_span(b, comp_len, d, key_batch_stride, key_row_stride) : 0;
    a.n_gather = n_gather;
    a.gather_out = static_cast<uint16_t *>(gather_out);
    if (p.ws_bytes > 0) {
        // arrival counters start at zero on every launch, whatever the workspace held before
        const cudaError_t e = cudaMemsetAsync(workspace, 0, static_cast<size_t>(a.ws_counter_bytes),
                                              static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return SEL_ECUDA;
    }
    return status_of(sel::launch_topk(dtype == SEL_F32 ? 0 : 1, p.mode, p.threads, n_gather > 0, p.smem, a, p.grid,
                                      static_cast<cudaStream_t>(stream)));
}

}  // namespace

namespace sel {

int check_topk_call(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride, int k, int sorted_index,
                    int idx_dtype, int want_values, const void *out_idx, int64_t out_idx_stride, const void *out_val,
                    int64_t out_val_stride)
{
    if (sorted_index < SEL_UNSORTED || sorted_index > SEL_SORT_VALUE) return SEL_EINVAL;
    return check_topk_args(x, dtype, rows, cols, stride, k, idx_dtype, want_values, out_idx, out_idx_stride, out_val,
                           out_val_stride, true);
}

}  // namespace sel

extern "C" {

int sel_set_tuning(int knob, int value)
{
    Tuning &t = tuning();
    switch (knob) {
    case SEL_TUNE_PLAN:
        if (value < SEL_PLAN_AUTO || value > SEL_PLAN_FLAT) return SEL_EINVAL;
        t.plan = value;
        return SEL_OK;
    case SEL_TUNE_PARTS:
        if (value < 0) return SEL_EINVAL;
        t.parts = value;
        return SEL_OK;
    case SEL_TUNE_ROW_SAMPLE:
        t.row_sample = value ? 1 : 0;
        return SEL_OK;
    case SEL_TUNE_HIST_AGG:
        t.hist_agg = value ? 1 : 0;
        return SEL_OK;
    case SEL_TUNE_ROW_ORDER:
        t.row_order = value ? 1 : 0;
        return SEL_OK;
    default: return SEL_EINVAL;
    }
}

int sel_get_tuning(int knob)
{
    Tuning &t = tuning();
    switch (knob) {
    case SEL_TUNE_PLAN: return t.plan.load();
    case SEL_TUNE_PARTS: return t.parts.load();
    case SEL_TUNE_ROW_SAMPLE: return t.row_sample.load();
    case SEL_TUNE_HIST_AGG: return t.hist_agg.load();
    case SEL_TUNE_ROW_ORDER: return t.row_order.load();
    default: return -1;
    }
}

int sel_debug_build(void)
{
#ifdef SEL_DEBUG
    return 1;
#else
    return 0;
#endif
}

int sel_selftest_wait_timeout(int32_t *err_flag, long long cycles, void *stream)
{
    if (!err_flag || cycles < 0) return SEL_EINVAL;
    return status_of(sel::launch_wait_selftest(err_flag, cycles, static_cast<cudaStream_t>(stream)));
}

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
    case SEL_ESCRATCH: return "shape needs more scratch than sel_topk_noalloc's built-in array (use sel_topk with a workspace)";
    case SEL_EBOUNDS: return "an out-of-bounds access was caught and skipped (debug build)";
    default: return "unknown status";
    }
}

int64_t sel_max_cols(int dtype)
{
    if (dtype != SEL_F32 && dtype != SEL_BF16) return 0;
    return 0x7fffffffLL;  // wider rows than one CTA can stage run split or streamed; indices are int32-safe
}

size_t sel_topk_workspace_size(int dtype, int64_t rows, int64_t cols, int k)
{
    if ((dtype != SEL_F32 && dtype != SEL_BF16) || rows <= 0 || cols < 0 || k < 1 || k > SEL_MAX_K) return 0;
    Plan p;
    if (cached_plan(dtype, rows, cols, k, false, 0, p) != SEL_OK) return 0;
    return p.ws_bytes;
}

const char *sel_topk_kernel_name(int dtype, int64_t rows, int64_t cols, int k, int64_t n_gather)
{
    if ((dtype != SEL_F32 && dtype != SEL_BF16) || rows <= 0 || cols < 0 || k < 1 || k > SEL_MAX_K) return nullptr;
    if (n_gather < 0 || n_gather > k) return nullptr;
    Plan p;
    if (cached_plan(dtype, rows, cols, k, n_gather > 0, n_gather, p) != SEL_OK) return nullptr;
    switch (p.mode) {
    case sel::kModeRow:
    case sel::kModeRowOrdered: return "row_kernel";
    case sel::kModeSplit: return "split_kernel";
    case sel::kModeWide:
    case sel::kModeWideSplit: return "wide_kernel";
    case sel::kModeStream: return "stream_kernel";
    case sel::kModeReg2:
    case sel::kModeReg8:
    case sel::kModeReg2Ordered:
    case sel::kModeReg8Ordered: return "reg_kernel";
    case sel::kModeFlat: return "flat_kernel";
    default: return nullptr;
    }
}

int sel_topk(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride, const int32_t *row_end, int k,
             int sorted_index, int idx_dtype, int want_values, void *out_idx, int64_t out_idx_stride, void *out_val,
             int64_t out_val_stride, void *workspace, size_t workspace_bytes, int32_t *nan_flag, int32_t *err_flag,
             void *stream)
{
    // The ordered compaction always yields ascending column order: SEL_SORT_INDEX costs nothing.
    if (sorted_index < SEL_UNSORTED || sorted_index > SEL_SORT_VALUE) return SEL_EINVAL;
    const int st = check_topk_args(x, dtype, rows, cols, stride, k, idx_dtype, want_values, out_idx, out_idx_stride,
                                   out_val, out_val_stride, true);
    if (st != SEL_OK || rows == 0) return st;
    // value order: ranked inside the staged row kernel where it can, else a second launch
    bool fused = sorted_index == SEL_SORT_VALUE;
    if (fused) {
        const int rc = run_topk(x, dtype, rows, cols, stride, row_end, k, idx_dtype, want_values, out_idx,
                                out_idx_stride, out_val, out_val_stride, nullptr, 1, 0, 0, 0, 0, 0, nullptr, workspace,
                                workspace_bytes, nan_flag, err_flag, stream, 1, &fused);
        if (rc != SEL_OK || fused) return rc;
    }
    const int rc = run_topk(x, dtype, rows, cols, stride, row_end, k, idx_dtype, want_values, out_idx, out_idx_stride,
                            out_val, out_val_stride, nullptr, 1, 0, 0, 0, 0, 0, nullptr, workspace, workspace_bytes,
                            nan_flag, err_flag, stream);
    if (rc != SEL_OK || sorted_index != SEL_SORT_VALUE) return rc;
    return value_order(x, dtype, rows, stride, k, idx_dtype, want_values, out_idx, out_idx_stride, out_val,
                       out_val_stride, stream);
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
    a.key_span = key_span(b, comp_len, d, key_batch_stride, key_row_stride);
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

int sel_gather_rows_pair(const void *key, int64_t d, int64_t key_batch_stride, int64_t key_row_stride,
                         const void *key2, int64_t d2, int64_t key2_batch_stride, int64_t key2_row_stride, int64_t b,
                         int64_t comp_len, const void *idx, int idx_dtype, int64_t rows, int64_t n,
                         int64_t idx_row_stride, void *out, void *out2, int32_t *err_flag, void *stream)
{
    if (idx_dtype != SEL_I32 && idx_dtype != SEL_I64) return SEL_EINVAL;
    if (n < 0 || rows < 0) return SEL_EINVAL;
    if (rows == 0 || n == 0) return (b >= 1 && rows % (b > 0 ? b : 1) == 0) ? SEL_OK : SEL_EINVAL;
    int st = check_gather_key(key, b, comp_len, d, key_batch_stride, key_row_stride, rows, out);
    if (st != SEL_OK) return st;
    st = check_gather_key(key2, b, comp_len, d2, key2_batch_stride, key2_row_stride, rows, out2);
    if (st != SEL_OK) return st;
    if (!idx || idx_row_stride < n) return SEL_EINVAL;
    sel::GatherArgs a{};
    a.key = static_cast<const uint16_t *>(key);
    a.comp_len = comp_len;
    a.d = d;
    a.key_batch_stride = key_batch_stride;
    a.key_row_stride = key_row_stride;
    a.key2 = static_cast<const uint16_t *>(key2);
    a.d2 = d2;
    a.key2_batch_stride = key2_batch_stride;
    a.key2_row_stride = key2_row_stride;
    a.key_span = key_span(b, comp_len, d, key_batch_stride, key_row_stride);
    a.key2_span = key_span(b, comp_len, d2, key2_batch_stride, key2_row_stride);
    a.out2 = static_cast<uint16_t *>(out2);
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

int sel_block_topk_gather(const void *scores, int dtype, int64_t rows, int64_t n_blocks, int64_t stride,
                          const int32_t *pos_end, int topk_blocks, int64_t block_size, int32_t *out_pos,
                          int64_t out_pos_stride, const void *key, int64_t b, int64_t comp_len, int64_t d,
                          int64_t key_batch_stride, int64_t key_row_stride, void *gather_out, void *workspace,
                          size_t workspace_bytes, int32_t *nan_flag, int32_t *err_flag, void *stream)
{
    if (block_size < 1 || n_blocks < 0) return SEL_EINVAL;
    if (n_blocks > 0 && n_blocks > 0x7fffffffLL / block_size) return SEL_EUNSUPPORTED;  // positions are int32
    if (topk_blocks >= 1 && static_cast<int64_t>(topk_blocks) * block_size > 0x7fffffffLL) return SEL_EUNSUPPORTED;
    int st = check_topk_args(scores, dtype, rows, n_blocks, stride, topk_blocks, SEL_I32, 0, out_pos,
                             out_pos_stride, nullptr, 0, true);
    if (st != SEL_OK) return st;
    const int64_t npos = static_cast<int64_t>(topk_blocks) * block_size;
    if (rows > 0 && out_pos_stride < npos) return SEL_EINVAL;
    if (key || gather_out) {
        st = check_gather_key(key, b, comp_len, d, key_batch_stride, key_row_stride, rows, gather_out);
        if (st != SEL_OK) return st;
    }
    if (rows == 0) return SEL_OK;
    sel::BlockArgs a{};
    if (n_blocks <= sel::kBlockSelectMax) {
        // few blocks a row: the expansion kernel selects them itself (one launch)
        a.scores = scores;
        a.scores_bf16 = dtype == SEL_BF16;
        a.n_blocks = n_blocks;
        a.scores_stride = stride;
        a.nan_flag = nan_flag;
    } else {
        // the selected block ids land in the first topk_blocks columns of out_pos (ascending, fills
        // last), to be expanded in place
        st = run_topk(scores, dtype, rows, n_blocks, stride, pos_end, topk_blocks, SEL_I32, 0, out_pos,
                      out_pos_stride, nullptr, 0, nullptr, 1, 0, 0, 0, 0, 0, nullptr, workspace, workspace_bytes,
                      nan_flag, err_flag, stream, block_size);
        if (st != SEL_OK) return st;
    }
    a.pos = out_pos;
    a.pos_stride = out_pos_stride;
    a.rows = rows;
    a.topk_blocks = topk_blocks;
    a.block_size = block_size;
    a.pos_end = pos_end;
    a.pos_limit = n_blocks * block_size;
    a.key = static_cast<const uint16_t *>(key);
    a.comp_len = comp_len;
    a.d = d;
    a.key_batch_stride = key_batch_stride;
    a.key_row_stride = key_row_stride;
    a.rows_per_batch = key ? rows / b : 1;
    a.key_span = key ? key_span(b, comp_len, d, key_batch_stride, key_row_stride) : 0;
    a.out = static_cast<uint16_t *>(gather_out);
    a.err_flag = err_flag;
    return status_of(sel::launch_block_expand(a, static_cast<cudaStream_t>(stream)));
}

int sel_topk_gather(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride, const int32_t *row_end,
                    int k, int sorted_index, int idx_dtype, int want_values, void *out_idx, int64_t out_idx_stride,
                    void *out_val, int64_t out_val_stride, const void *key, int64_t b, int64_t comp_len, int64_t d,
                    int64_t key_batch_stride, int64_t key_row_stride, int64_t n_gather, void *gather_out,
                    void *workspace, size_t workspace_bytes, int32_t *nan_flag, int32_t *err_flag, void *stream)
{
    if (sorted_index < SEL_UNSORTED || sorted_index > SEL_SORT_VALUE) return SEL_EINVAL;
    const bool by_value = sorted_index == SEL_SORT_VALUE;
    int st = check_topk_args(x, dtype, rows, cols, stride, k, idx_dtype, want_values, out_idx, out_idx_stride, out_val,
                             out_val_stride, by_value);
    if (st != SEL_OK) return st;
    if (n_gather < 0 || n_gather > k) return SEL_EINVAL;
    if (rows == 0) return (b >= 1) ? SEL_OK : SEL_EINVAL;
    if (n_gather > 0) {
        st = check_gather_key(key, b, comp_len, d, key_batch_stride, key_row_stride, rows, gather_out);
        if (st != SEL_OK) return st;
    }
    if (by_value) {
        // the staged row kernel ranks, writes and gathers in one launch where it can; else the
        // selection, then one launch that orders the rows and gathers the first n_gather ordered
        // columns' key rows
        bool fused = true;
        st = run_topk(x, dtype, rows, cols, stride, row_end, k, idx_dtype, want_values, out_idx, out_idx_stride,
                      out_val, out_val_stride, key, n_gather > 0 ? b : 1, comp_len, d, key_batch_stride,
                      key_row_stride, n_gather, gather_out, workspace, workspace_bytes, nan_flag, err_flag, stream, 1,
                      &fused);
        if (st != SEL_OK || fused) return st;
        st = run_topk(x, dtype, rows, cols, stride, row_end, k, idx_dtype, want_values, out_idx, out_idx_stride,
                      out_val, out_val_stride, nullptr, 1, 0, 0, 0, 0, 0, nullptr, workspace, workspace_bytes,
                      nan_flag, err_flag, stream);
        if (st != SEL_OK) return st;
        OrderGather g;
        if (n_gather > 0) {
            g.key = key;
            g.b = b;
            g.comp_len = comp_len;
            g.d = d;
            g.key_batch_stride = key_batch_stride;
            g.key_row_stride = key_row_stride;
            g.n_gather = n_gather;
            g.gather_out = gather_out;
            g.err_flag = err_flag;
        }
        return value_order(x, dtype, rows, stride, k, idx_dtype, want_values, out_idx, out_idx_stride, out_val,
                           out_val_stride, stream, g);
    }
    return run_topk(x, dtype, rows, cols, stride, row_end, k, idx_dtype, want_values, out_idx, out_idx_stride, out_val,
                    out_val_stride, key, n_gather > 0 ? b : 1, comp_len, d, key_batch_stride, key_row_stride, n_gather,
                    gather_out, workspace, workspace_bytes, nan_flag, err_flag, stream);
}

}  // extern "C"
