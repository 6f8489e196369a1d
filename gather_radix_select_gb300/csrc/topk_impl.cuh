// topk_impl.cuh -- batched row-wise top-k by radix select, with an optional
// fused gather of the selected key rows.
//
// What is computed ("Speed up PyTorch TopK with DeepSelect": "Basic TopK
// usage", "Working with variable-length rows", "NaN handling"): for each row
// r with n = clamp(row_end[r], 0, cols) valid columns, the k largest values
// (ties: smaller column first), or, when n <= k, every valid column followed
// by fills (index -1, value -inf).  Rows with n > k are checked for NaN.
//
// Six kernels, chosen per launch by the host plan:
//   reg_kernel    one CTA per row of at most 16 KB; the row is held in
//                 registers (a contiguous run of vectors per thread) and the
//                 radix levels run from there.
//   row_kernel    one CTA per row; the row is staged whole in shared memory.
//   wide_kernel   rows too wide to stage: each warp streams its share of the
//                 row with 16-byte loads (read once), tests every vector
//                 against a threshold estimated from the first loads, and
//                 appends the passing keys to its own region of a candidate
//                 list in shared memory; the selection runs on the regions.
//                 Few wide rows are cut into parts whose candidates meet in a
//                 caller workspace, merged by the last part to arrive.
//   split_kernel  a wide row is cut into `parts` slices, one CTA each.  Every
//                 CTA filters its slice down to an index-ordered candidate
//                 list in a caller-provided workspace; the CTA that finishes
//                 last (an atomic arrival counter -- nobody waits) selects
//                 the k from the merged candidates.
//   stream_kernel one CTA per row, the row read from global memory on every
//                 radix pass (the exact fallback of the others).
//   flat_kernel   rows cut into chunks dealt over one resident CTA per SM;
//                 streaming warps filter, helper warps estimate, flush and
//                 select (reached only when forced: measured slower, see the
//                 kernel's comment).
//
// Building blocks (GB300 design):
//   * Staged slices (row_kernel, split_kernel) arrive in shared memory by bulk
//     async copies (cp.async.bulk, 16 KB chunks, one mbarrier each); waiting
//     threads sleep in hardware (try_wait with a suspend hint), bounded by a
//     ~2 s budget.
//   * Order-preserving key: fp32/bf16 bits -> unsigned key, larger float =>
//     larger key, -0 folded onto +0.
//   * Radix select over digits from the most significant end (11/11/10 bits
//     fp32, 11/5 bf16, 8/8 for short bf16 rows); histograms in shared memory.
//   * First digit: exact histogram while chunks land, or, for long rows, the
//     histogram of every 8th 16-byte vector, from which a threshold digit is
//     estimated with a margin; one pass then filters the keys at or above it
//     into an index-ordered candidate list (mask byte per vector + block
//     scan).  Too few candidates is detected and repaired exactly.
//   * A level stops early when the threshold bin holds exactly the keys
//     still needed.
//   * Compaction is ordered: keys above the threshold class are all taken,
//     keys in it are taken in column order until k are chosen (block scans
//     give tie ranks and output positions).  Output rows therefore come in
//     ascending column order and sorted_index costs nothing.
#pragma once

#include <cstdint>

#include "ptx.cuh"
#include "order_core.cuh"
#include "sel_internal.h"

namespace sel {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr long long kWaitCycles = 4000000000LL;  // bound on any mbarrier wait (~2 s)
constexpr int32_t kStatusInval = 1;
constexpr int32_t kStatusTimeout = 5;

// A set of consecutive warps that synchronises on its own: the whole CTA (barrier 0, i.e.
// __syncthreads), or warps [BASE/32, (BASE+NT)/32) on named barrier BAR.  Helpers that run on
// a group use G::tid() (0..NT-1 within the group) and G::sync() instead of threadIdx.x and
// __syncthreads().
template <int NT_, int BAR = 0, int BASE = 0>
struct Grp {
    static constexpr int NT = NT_;
    static constexpr int W = NT_ / 32;
    static_assert(NT_ % 32 == 0 && BASE % 32 == 0, "whole warps");
    static __device__ __forceinline__ int tid() { return static_cast<int>(threadIdx.x) - BASE; }
    static __device__ __forceinline__ void sync()
    {
        if constexpr (BAR == 0)
            __syncthreads();
        else
            asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT_) : "memory");
    }
    // sync() that also returns whether `p` held on any thread of the group
    static __device__ __forceinline__ bool sync_or(bool p)
    {
        if constexpr (BAR == 0) {
            return __syncthreads_or(p) != 0;
        } else {
            uint32_t r;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                : "=r"(r)
                : "r"(static_cast<uint32_t>(p)), "n"(BAR), "n"(NT_)
                : "memory");
            return r != 0;
        }
    }
};

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
    static constexpr uint32_t kInfMagnitude = 0x7f800000u;
    static __device__ __forceinline__ uint32_t magnitude(uint32_t u) { return u & 0x7fffffffu; }
    static __device__ __forceinline__ bool is_nan(uint32_t u) { return (u & 0x7fffffffu) > 0x7f800000u; }
    static constexpr uint32_t kSignKey = 0x80000000u;  // key of +0 and -0
    // Bit t set when key(element t) >= tkey, for a threshold above +/-0 (tkey > kSignKey), where
    // that is a signed compare of the raw bits with ts = tkey ^ kSignKey; folds |x| into mag.
    static __device__ __forceinline__ uint32_t ge_mask_positive(const uint4 &q, uint32_t ts, uint32_t &mag)
    {
        const int t = static_cast<int>(ts);
        mag = max(mag, max(max(q.x & 0x7fffffffu, q.y & 0x7fffffffu), max(q.z & 0x7fffffffu, q.w & 0x7fffffffu)));
        return static_cast<uint32_t>(static_cast<int>(q.x) >= t) | (static_cast<uint32_t>(static_cast<int>(q.y) >= t) << 1) |
               (static_cast<uint32_t>(static_cast<int>(q.z) >= t) << 2) |
               (static_cast<uint32_t>(static_cast<int>(q.w) >= t) << 3);
    }
    // NaN detection on raw words without per-element work: a positive NaN is the largest signed
    // pattern (> 0x7f800000), a negative NaN the largest unsigned one (> 0xff800000).
    static constexpr uint32_t kSmaxInit = 0x80000000u, kUmaxInit = 0u;
    static __device__ __forceinline__ void nan_acc(const uint4 &q, uint32_t &smax, uint32_t &umax)
    {
        const int m = max(max(static_cast<int>(q.x), static_cast<int>(q.y)), max(static_cast<int>(q.z), static_cast<int>(q.w)));
        smax = static_cast<uint32_t>(max(static_cast<int>(smax), m));
        umax = max(umax, max(max(q.x, q.y), max(q.z, q.w)));
    }
    static __device__ __forceinline__ void nan_acc1(uint32_t u, uint32_t &smax, uint32_t &umax)
    {
        smax = static_cast<uint32_t>(max(static_cast<int>(smax), static_cast<int>(u)));
        umax = max(umax, u);
    }
    static __device__ __forceinline__ bool has_nan(uint32_t smax, uint32_t umax)
    {
        return static_cast<int>(smax) > 0x7f800000 || umax > 0xff800000u;
    }
    // As ge_mask_positive, without the magnitude.
    static __device__ __forceinline__ uint32_t ge_mask_raw(const uint4 &q, uint32_t ts)
    {
        const int t = static_cast<int>(ts);
        return static_cast<uint32_t>(static_cast<int>(q.x) >= t) | (static_cast<uint32_t>(static_cast<int>(q.y) >= t) << 1) |
               (static_cast<uint32_t>(static_cast<int>(q.z) >= t) << 2) |
               (static_cast<uint32_t>(static_cast<int>(q.w) >= t) << 3);
    }
    // Bit t set when key(element t) >= tkey (any threshold).
    static __device__ __forceinline__ uint32_t ge_mask_key(const uint4 &q, uint32_t tkey)
    {
        return static_cast<uint32_t>(key(q.x) >= tkey) | (static_cast<uint32_t>(key(q.y) >= tkey) << 1) |
               (static_cast<uint32_t>(key(q.z) >= tkey) << 2) | (static_cast<uint32_t>(key(q.w) >= tkey) << 3);
    }
    // element t (0..3) of a vector
    static __device__ __forceinline__ uint32_t lane_of(const uint4 &q, int t)
    {
        const uint32_t lo = (t & 1) ? q.y : q.x, hi = (t & 1) ? q.w : q.z;
        return (t & 2) ? hi : lo;
    }
    static __device__ __forceinline__ void unpack(const uint4 &q, uint32_t (&e)[4])
    {
        e[0] = q.x;
        e[1] = q.y;
        e[2] = q.z;
        e[3] = q.w;
    }
    static __device__ __forceinline__ uint4 pack(const uint32_t (&e)[4]) { return make_uint4(e[0], e[1], e[2], e[3]); }
    // Streaming test with running maxima: smax_vec = signed maximum of a vector's raw words; a
    // vector holds a key >= tkey (threshold above +/-0, ts = tkey ^ kSignKey) iff ge_raw(smax_vec,
    // ts).  smax_fold / umax_fold keep the running signed / unsigned maxima that has_nan reads;
    // smax_key is the key of the largest element folded into a running signed maximum.
    static __device__ __forceinline__ uint32_t smax_vec(const uint4 &q)
    {
        return static_cast<uint32_t>(max(__vimax3_s32(static_cast<int>(q.x), static_cast<int>(q.y), static_cast<int>(q.z)),
                                         static_cast<int>(q.w)));
    }
    static __device__ __forceinline__ uint32_t smax_fold(uint32_t s, uint32_t ms)
    {
        return static_cast<uint32_t>(max(static_cast<int>(s), static_cast<int>(ms)));
    }
    static __device__ __forceinline__ uint32_t umax_fold(uint32_t u, const uint4 &q)
    {
        return __vimax3_u32(u, __vimax3_u32(q.x, q.y, q.z), q.w);
    }
    static __device__ __forceinline__ bool ge_raw(uint32_t ms, uint32_t ts) { return static_cast<int>(ms) >= static_cast<int>(ts); }
    static __device__ __forceinline__ uint32_t smax_key(uint32_t s) { return key(s); }
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
    static constexpr uint32_t kInfMagnitude = 0x7f80u;
    static __device__ __forceinline__ uint32_t magnitude(uint16_t h) { return h & 0x7fffu; }
    static __device__ __forceinline__ bool is_nan(uint16_t h) { return (h & 0x7fffu) > 0x7f80u; }
    static constexpr uint32_t kSignKey = 0x8000u;  // key of +0 and -0
    // As for fp32, on the two 16-bit halves of each word (element 2i low, 2i+1 high).
    static __device__ __forceinline__ uint32_t ge_mask_positive(const uint4 &q, uint32_t ts, uint32_t &mag)
    {
        const int t = static_cast<int>(ts << 16);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t m = 0, mm = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m |= static_cast<uint32_t>(static_cast<int>(w[i] << 16) >= t) << (2 * i);
            m |= static_cast<uint32_t>(static_cast<int>(w[i] & 0xffff0000u) >= t) << (2 * i + 1);
            mm = __vmaxu2(mm, w[i] & 0x7fff7fffu);
        }
        mag = max(mag, max(mm & 0xffffu, mm >> 16));
        return m;
    }
    // As for fp32, per 16-bit half: a positive NaN half is the largest signed half (> 0x7f80), a
    // negative NaN half the largest unsigned one (> 0xff80).
    static constexpr uint32_t kSmaxInit = 0x80008000u, kUmaxInit = 0u;
    static __device__ __forceinline__ void nan_acc(const uint4 &q, uint32_t &smax, uint32_t &umax)
    {
        smax = __vmaxs2(smax, __vmaxs2(__vmaxs2(q.x, q.y), __vmaxs2(q.z, q.w)));
        umax = __vmaxu2(umax, __vmaxu2(__vmaxu2(q.x, q.y), __vmaxu2(q.z, q.w)));
    }
    static __device__ __forceinline__ void nan_acc1(uint16_t h, uint32_t &smax, uint32_t &umax)
    {
        smax = __vmaxs2(smax, static_cast<uint32_t>(h) | 0x80000000u);  // other half: the signed minimum
        umax = __vmaxu2(umax, static_cast<uint32_t>(h));
    }
    static __device__ __forceinline__ bool has_nan(uint32_t smax, uint32_t umax)
    {
        return static_cast<int16_t>(smax & 0xffffu) > 0x7f80 || static_cast<int16_t>(smax >> 16) > 0x7f80 ||
               (umax & 0xffffu) > 0xff80u || (umax >> 16) > 0xff80u;
    }
    static __device__ __forceinline__ uint32_t ge_mask_raw(const uint4 &q, uint32_t ts)
    {
        const int t = static_cast<int>(ts << 16);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m |= static_cast<uint32_t>(static_cast<int>(w[i] << 16) >= t) << (2 * i);
            m |= static_cast<uint32_t>(static_cast<int>(w[i] & 0xffff0000u) >= t) << (2 * i + 1);
        }
        return m;
    }
    static __device__ __forceinline__ uint32_t ge_mask_key(const uint4 &q, uint32_t tkey)
    {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m |= static_cast<uint32_t>(key(static_cast<uint16_t>(w[i] & 0xffffu)) >= tkey) << (2 * i);
            m |= static_cast<uint32_t>(key(static_cast<uint16_t>(w[i] >> 16)) >= tkey) << (2 * i + 1);
        }
        return m;
    }
    // element t (0..7) of a vector
    static __device__ __forceinline__ uint16_t lane_of(const uint4 &q, int t)
    {
        const uint32_t lo = (t & 2) ? q.y : q.x, hi = (t & 2) ? q.w : q.z;
        const uint32_t w = (t & 4) ? hi : lo;
        return static_cast<uint16_t>((t & 1) ? (w >> 16) : (w & 0xffffu));
    }
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
    static __device__ __forceinline__ uint4 pack(const uint16_t (&e)[8])
    {
        return make_uint4(e[0] | (static_cast<uint32_t>(e[1]) << 16), e[2] | (static_cast<uint32_t>(e[3]) << 16),
                          e[4] | (static_cast<uint32_t>(e[5]) << 16), e[6] | (static_cast<uint32_t>(e[7]) << 16));
    }
    // As for fp32, on the two 16-bit halves of each word (packed per-half maxima).
    static __device__ __forceinline__ uint32_t smax_vec(const uint4 &q) { return __vmaxs2(__vimax3_s16x2(q.x, q.y, q.z), q.w); }
    static __device__ __forceinline__ uint32_t smax_fold(uint32_t s, uint32_t ms) { return __vmaxs2(s, ms); }
    static __device__ __forceinline__ uint32_t umax_fold(uint32_t u, const uint4 &q)
    {
        return __vimax3_u16x2(u, __vimax3_u16x2(q.x, q.y, q.z), q.w);
    }
    static __device__ __forceinline__ bool ge_raw(uint32_t ms, uint32_t ts)
    {
        const int t = static_cast<int>(ts << 16);
        return static_cast<int>(ms << 16) >= t || static_cast<int>(ms & 0xffff0000u) >= t;
    }
    static __device__ __forceinline__ uint32_t smax_key(uint32_t s)
    {
        const int16_t lo = static_cast<int16_t>(s & 0xffffu), hi = static_cast<int16_t>(s >> 16);
        return key(static_cast<uint16_t>(lo > hi ? lo : hi));
    }
};

__device__ __forceinline__ void set_err(int32_t *flag, int32_t code)
{
    if (flag) atomicCAS(flag, 0, code);
}

// Bounded wait on an mbarrier phase: after `budget` clock cycles (~2 s by default) the wait gives
// up, records a timeout in err_flag and lets the CTA run on (its results are then unspecified).
__device__ __forceinline__ void wait_phase(uint64_t *bar, uint32_t parity, int32_t *err,
                                           long long budget = kWaitCycles)
{
    constexpr uint32_t kSuspendNs = 100000;  // each try sleeps in hardware for up to 0.1 ms
    if (mbar_try_wait(bar, parity, kSuspendNs)) return;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity, kSuspendNs)) {
        if (clock64() - t0 > budget) {
            set_err(err, kStatusTimeout);
            return;
        }
    }
}

// Prefetches [p, p + bytes) into L2 (p and bytes multiples of 16); no registers held, nothing waited for.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Warp-aggregated shared histogram increment: lanes with equal digits are grouped with
// __match_any_sync and only the group leader adds the group's size.  For digits that pile
// up on few bins (candidates near the threshold, tie-heavy classes).  All 32 lanes must call.
__device__ __forceinline__ void hist_add_grouped(uint32_t *hist, uint32_t digit, bool valid, int lane)
{
    const unsigned peers = __match_any_sync(kFull, valid ? digit : 0xffffffffu);
    if (valid && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(peers)));
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

// Exclusive prefix sum over the group (thread order); `total` gets the group's sum.
// Uses s_warp[G::W]; contains two group barriers.
template <typename G>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *s_warp, uint32_t &total)
{
    constexpr int NT = G::NT;
    const int lane = G::tid() & 31, warp = G::tid() >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) s_warp[warp] = inc;
    G::sync();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const uint32_t t = s_warp[w];
        before += (w < warp) ? t : 0u;
        tot += t;
    }
    G::sync();
    total = tot;
    return before + inc - v;
}

// Threshold digit of a histogram h[0, nb): the digit d with
//   sum_{e > d} h[e] < need <= sum_{e >= d} h[e].
// Result in out[0] = d, out[1] = sum_{e > d} h[e], out[2] = h[d].  Every thread of the group calls.
template <typename G>
__device__ void find_threshold(const uint32_t *h, int nb, uint32_t need, uint32_t *out, uint32_t *s_warp)
{
    constexpr int NT = G::NT;
    const int tid = G::tid();
    const int per = nb > NT ? nb / NT : 1;
    const int lo = tid * per;
    uint32_t s = 0;
    if (lo < nb) {
        // each thread sums its `per` consecutive bins starting at a rotated bin, so that the
        // threads of a warp read distinct banks (per is a power of two)
        const int rot = (tid * per / 32) & (per - 1);
        for (int i = 0; i < per; ++i) s += h[lo + ((i + rot) & (per - 1))];
    }
    // exclusive scan in reversed thread order gives the count above this thread's bins
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t inc = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(kFull, inc, o);
        if (lane + o < 32) inc += y;
    }
    if (lane == 0) s_warp[warp] = inc;
    G::sync();
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
    G::sync();
}

__device__ __forceinline__ void store_idx(const TopkArgs &a, int64_t row, int64_t pos, int64_t col)
{
    if (!a.out_idx) return;
    if (!SEL_IN_BOUNDS(row >= 0 && row < a.rows && pos >= 0 && pos < a.k, a.err_flag)) return;
    if (a.idx_i64)
        static_cast<int64_t *>(a.out_idx)[row * a.out_idx_stride + pos] = col;
    else
        static_cast<int32_t *>(a.out_idx)[row * a.out_idx_stride + pos] = static_cast<int32_t>(col);
}

template <typename E>
__device__ __forceinline__ void store_val(const TopkArgs &a, int64_t row, int64_t pos, E v)
{
    if (!SEL_IN_BOUNDS(row >= 0 && row < a.rows && pos >= 0 && pos < a.k, a.err_flag)) return;
    static_cast<E *>(a.out_val)[row * a.out_val_stride + pos] = v;
}

// Copies key rows for output positions [j0, j1) of `row`:
//   gather_out[row, j, :] = key[row / rows_per_batch, max(col_j, 0), :]
// col_j = glist[j - j0] when glist is given, else j for j < n_short and 0 beyond.
template <typename G>
__device__ void gather_rows_of(const TopkArgs &a, int64_t row, int64_t j0, int64_t j1, const int32_t *glist,
                               int64_t n_short)
{
    constexpr int NT = G::NT;
    const int gt = G::tid();
    const int vpr = static_cast<int>(a.d >> 3);  // 16-byte vectors per key row
    const int vsh = (vpr & (vpr - 1)) == 0 ? __ffs(vpr) - 1 : -1;  // log2(vpr), or -1
    const int64_t bb = row / a.rows_per_batch;
    const uint16_t *kb = a.key + bb * a.key_batch_stride;
    uint4 *ob = reinterpret_cast<uint4 *>(a.gather_out + (row * a.n_gather + j0) * a.d);
    const int total = static_cast<int>(j1 - j0) * vpr;
    constexpr int U = 4;
    if (vsh >= 1 && vpr <= 2 * NT) {
        // rows of a power-of-two number (>= 2) of vectors: lpr = vpr / 2 lanes share a row and
        // thread t copies vectors c and c + lpr (c = t mod lpr) of rows t / lpr, t / lpr + NT / lpr,
        // ... -- a row's column is read once for two vectors, no index division, and each load or
        // store instruction covers whole 128-byte pieces of the rows
        const int nrows = static_cast<int>(j1 - j0);
        const int lsh = vsh - 1, lpr = vpr >> 1;
        const int c = gt & (lpr - 1);
        const int rstep = NT >> lsh;
        constexpr int UR = NT <= 128 ? U : U / 2;  // rows a thread has in flight (two vectors each)
        for (int jb = gt >> lsh; jb < nrows; jb += UR * rstep) {
            uint4 v[UR][2];
#pragma unroll
            for (int u = 0; u < UR; ++u) {
                const int jj = jb + u * rstep;
                v[u][0] = v[u][1] = make_uint4(0u, 0u, 0u, 0u);
                if (jj < nrows) {
                    const int64_t j = j0 + jj;
                    int64_t p = glist ? static_cast<int64_t>(glist[jj]) : (j < n_short ? j : 0);
                    if (p < 0) p = 0;
                    if (p < a.comp_len) {
                        const uint4 *src = reinterpret_cast<const uint4 *>(kb + p * a.key_row_stride) + c;
                        if (SEL_IN_BOUNDS(bb * a.key_batch_stride + p * a.key_row_stride + a.d <= a.key_span, a.err_flag)) {
                            v[u][0] = __ldg(src);
                            v[u][1] = __ldg(src + lpr);
                        }
                    } else if (c == 0) {
                        set_err(a.err_flag, kStatusInval);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < UR; ++u) {
                const int jj = jb + u * rstep;
                if (jj < nrows && SEL_IN_BOUNDS(row < a.rows && j0 + jj < a.n_gather, a.err_flag)) {
                    uint4 *dst = ob + (static_cast<int64_t>(jj) << vsh) + c;
                    __stcs(dst, v[u][0]);
                    __stcs(dst + lpr, v[u][1]);
                }
            }
        }
        return;
    }
    for (int t0 = gt; t0 < total; t0 += U * NT) {
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
                if (p < a.comp_len) {
                    if (SEL_IN_BOUNDS(bb * a.key_batch_stride + p * a.key_row_stride + a.d <= a.key_span, a.err_flag))
                        v[u] = __ldg(reinterpret_cast<const uint4 *>(kb + p * a.key_row_stride) + (t - jj * vpr));
                } else if (t - jj * vpr == 0)
                    set_err(a.err_flag, kStatusInval);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = t0 + u * NT;
            if (t < total && SEL_IN_BOUNDS(row < a.rows && j0 + t / vpr < a.n_gather, a.err_flag)) __stcs(ob + t, v[u]);
        }
    }
}

template <int NT>
struct MinBlocks {
    static constexpr int value = NT >= 512 ? 2 : (NT >= 256 ? 4 : 8);
};

// Short row (n <= k): columns 0..n-1 then fills; positions [j0, j1) of the output row.
template <typename E, typename G, bool GATHER>
__device__ void short_row(const TopkArgs &a, int64_t row, int64_t n, int j0, int j1)
{
    using T = Elem<E>;
    const E *xrow = static_cast<const E *>(a.x) + row * a.stride;
    for (int j = j0 + G::tid(); j < j1; j += G::NT) {
        store_idx(a, row, j, j < n ? j : -1);
        if (a.want_values) store_val<E>(a, row, j, j < n ? xrow[j] : static_cast<E>(T::kFill));
    }
    if (GATHER) {
        const int64_t g1 = min(static_cast<int64_t>(j1), a.n_gather);
        if (j0 < g1) gather_rows_of<G>(a, row, j0, g1, nullptr, n);
    }
}

// Row taken by CTA (or CTA group) b.  With per-row ends the rows' lengths often grow or shrink
// along the batch (causal masks), and launched in order the longest rows would all run in the
// last wave; row_order = 1 interleaves the two ends of the batch instead (b even: row b/2, b odd:
// row rows-1-b/2), so that every wave holds a mix (the dual-chunk assignment of the PaddleFleet
// pull request "Balance the latent-MQA indexer's CP rows with a dual-chunk swap", applied to
// CTAs).  A permutation of [0, rows).  Off by default: on the causal bf16 [4096, 2048] rows it
// measured slower (top-k 30.8 against 29.0 us): in order, neighbouring rows' traffic stays together.
__device__ __forceinline__ int64_t row_of_block(const TopkArgs &a, int64_t b)
{
    if (!a.row_order) return b;
    const int64_t h = b >> 1;
    return (b & 1) ? a.rows - 1 - h : h;
}

__device__ __forceinline__ int64_t valid_cols(const TopkArgs &a, int64_t row)
{
    int64_t n = a.cols;
    if (a.row_end) {
        int64_t re = a.row_end[row];
        // row_end in units of row_end_div columns' worth (block selection: a row end in positions,
        // a column per block; the blocks holding a valid position)
        if (a.row_end_div > 1) re = re <= 0 ? 0 : (re + a.row_end_div - 1) / a.row_end_div;
        n = re < 0 ? 0 : (re > a.cols ? a.cols : re);
    }
    return n;
}

// Stages xrow[lo, lo+len) into smem (bulk copies for the 16-byte part, plain loads for the rest)
// and adds every `step`-th 16-byte vector's top digits into hist while the chunks land.
// Returns after a __syncthreads; hist must be zero on entry.
template <typename E, int NT>
__device__ void stage_and_histogram(const TopkArgs &a, const E *xrow, int64_t lo, int len, int step,
                                    unsigned char *smem, uint32_t *hist, uint64_t *bars)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    E *buf = reinterpret_cast<E *>(smem);
    const uint32_t bytes = static_cast<uint32_t>(len) * sizeof(E);
    const uint32_t bulk = bytes & ~15u;
    const int nchunks = static_cast<int>((bulk + kChunkBytes - 1) / kChunkBytes);
    const bool agg = a.agg != 0;
    if (tid == 0) {
        for (int c = 0; c < nchunks; ++c) mbar_init(&bars[c], 1);
        fence_mbar_init();
        const char *src = reinterpret_cast<const char *>(xrow + lo);
        for (int c = 0; c < nchunks; ++c) {
            const uint32_t nb = min(kChunkBytes, bulk - static_cast<uint32_t>(c) * kChunkBytes);
            mbar_arrive_expect_tx(&bars[c], nb);
            bulk_load(smem + static_cast<size_t>(c) * kChunkBytes, src + static_cast<size_t>(c) * kChunkBytes, nb,
                      &bars[c]);
        }
    }
    __syncthreads();  // barriers initialised before anyone waits on them
    const int sh0 = T::KB - a.bits[0];
    for (int c = 0; c < nchunks; ++c) {
        wait_phase(&bars[c], 0u, a.err_flag);
        const uint32_t cb = min(kChunkBytes, bulk - static_cast<uint32_t>(c) * kChunkBytes);
        const int nv = static_cast<int>(cb >> 4);
        const uint4 *vb = reinterpret_cast<const uint4 *>(smem + static_cast<size_t>(c) * kChunkBytes);
        if (agg) {
            for (int base = warp * 32; base * step < nv; base += NT) {
                const int v = (base + lane) * step;
                const bool ok = v < nv;
                E el[V];
                T::unpack(ok ? vb[v] : make_uint4(0u, 0u, 0u, 0u), el);
#pragma unroll
                for (int t = 0; t < V; ++t) hist_add_grouped(hist, T::key(el[t]) >> sh0, ok, lane);
            }
        } else {
            for (int v = tid * step; v < nv; v += NT * step) {
                E el[V];
                T::unpack(vb[v], el);
#pragma unroll
                for (int t = 0; t < V; ++t) atomicAdd(&hist[T::key(el[t]) >> sh0], 1u);
            }
        }
    }
    const int tail0 = static_cast<int>(bulk / sizeof(E));
    if (tid < len - tail0) {  // < 16 bytes left over: plain loads
        const E e = xrow[lo + tail0 + tid];
        buf[tail0 + tid] = e;
        if (step == 1) atomicAdd(&hist[T::key(e) >> sh0], 1u);
    }
    __syncthreads();
}

// One pass over the staged slice: mask byte per 16-byte vector (bit t: key >= tkey), NaN check
// into nan_flag, then the index-ordered list of 16-bit offsets of the set bits.  Returns the
// number of such keys; the list is written only if that number is <= cap.  Ends with __syncthreads.
template <typename E, int NT>
__device__ int filter_to_list(const TopkArgs &a, const E *buf, int len, uint32_t tkey, uint8_t *masks, uint16_t *list,
                              int cap, uint32_t *s_warp)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nvt = (len + V - 1) / V;
    const uint4 *vbuf = reinterpret_cast<const uint4 *>(buf);
    uint32_t mag = 0;  // largest |x| bit pattern: a NaN iff above the infinity pattern
    const bool positive = tkey > T::kSignKey;  // raw-bit compare suffices above +/-0
    const uint32_t ts = tkey ^ T::kSignKey;
    const int nfull = len / V;                 // vectors with every element in range
    for (int base = warp * 32; base < nvt; base += NT) {
        const int v = base + lane;
        if (v < nvt) {
            const uint4 q = vbuf[v];
            uint32_t m = 0;
            if (positive && v < nfull) {
                m = T::ge_mask_positive(q, ts, mag);
            } else {
                E el[V];
                T::unpack(q, el);
                const int lim = min(V, len - v * V);
#pragma unroll
                for (int t = 0; t < V; ++t) {
                    const bool in = t < lim;
                    mag = max(mag, in ? T::magnitude(el[t]) : 0u);
                    m |= static_cast<uint32_t>(in && T::key(el[t]) >= tkey) << t;
                }
            }
            masks[v] = static_cast<uint8_t>(m);
        }
    }
    if (__syncthreads_or(mag > T::kInfMagnitude) && tid == 0 && a.nan_flag) atomicOr(a.nan_flag, 1);
    const int q = (nvt + NT - 1) / NT;
    const int v0 = min(nvt, tid * q), v1 = min(nvt, v0 + q);
    uint32_t c = 0;
    for (int v = v0; v < v1; ++v) c += __popc(static_cast<uint32_t>(masks[v]));
    uint32_t tot;
    uint32_t pos = block_exclusive_scan<Grp<NT>>(c, s_warp, tot);
    if (tot <= static_cast<uint32_t>(cap)) {
        for (int v = v0; v < v1; ++v) {
            uint32_t m = masks[v];
            while (m) {
                const int b = __ffs(m) - 1;
                if (SEL_IN_BOUNDS(v * V + b < len && pos < static_cast<uint32_t>(cap), a.err_flag))
                    list[pos] = static_cast<uint16_t>(v * V + b);
                ++pos;
                m &= m - 1u;
            }
        }
    }
    __syncthreads();
    return static_cast<int>(tot);
}

// Sum of a histogram over the CTA (all threads get it).  Two __syncthreads.
template <typename G>
__device__ __forceinline__ uint32_t hist_total(const uint32_t *h, int nb, uint32_t *s_warp)
{
    constexpr int NT = G::NT;
    const int tid = G::tid();
    uint32_t s = 0;
    for (int i = tid; i < nb; i += NT) s += h[i];
    s = __reduce_add_sync(kFull, s);
    if ((tid & 31) == 0) s_warp[tid >> 5] = s;
    G::sync();
    uint32_t total = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) total += s_warp[w];
    G::sync();
    return total;
}

// Threshold key estimated from a sample: every `step`-th of the first `nvb` full 16-byte vectors
// of buf, whose top-digit histogram is in h.  mu = the sample's expected share of the `share`
// keys wanted out of `population`; the estimate keeps mu*(1+1/8) + 3*sqrt(mu) + 4 sampled keys at
// or above it.  The top digit comes from h, a second digit from the sampled keys in that bin, so
// the key is resolved to 22 bits (fp32) or fully (bf16).  0 (keep everything) if that is the
// whole sample.  Leaves h zero.
template <typename E, int NT>
__device__ uint32_t sample_threshold_key(const TopkArgs &a, const E *buf, int nvb, int step, uint32_t *h,
                                         float share, float population, uint32_t *s_res, uint32_t *s_warp)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sh0 = T::KB - a.bits[0];
    const int nb0 = 1 << a.bits[0];
    const uint32_t total = hist_total<Grp<NT>>(h, nb0, s_warp);
    const float mu = share * static_cast<float>(total) / population;
    const float want = mu * 1.125f + 3.0f * sqrtf(mu) + 4.0f;
    if (want >= static_cast<float>(total)) {
        for (int i = tid; i < nb0; i += NT) h[i] = 0u;
        __syncthreads();
        return 0u;
    }
    find_threshold<Grp<NT>>(h, nb0, static_cast<uint32_t>(want), s_res, s_warp);
    const uint32_t d = s_res[0];
    const uint32_t need2 = static_cast<uint32_t>(want) - s_res[1];
    for (int i = tid; i < nb0; i += NT) h[i] = 0u;
    __syncthreads();
    const int b2 = sh0 < 11 ? sh0 : 11;  // refinement digit: the next bits below the top digit
    const int sh1 = sh0 - b2;
    const uint32_t m2 = (1u << b2) - 1u;
    const uint4 *vb = reinterpret_cast<const uint4 *>(buf);
    for (int base = warp * 32; base * step < nvb; base += NT) {
        const int v = (base + lane) * step;
        if (v < nvb) {
            E el[V];
            T::unpack(vb[v], el);
#pragma unroll
            for (int t = 0; t < V; ++t) {
                const uint32_t kk = T::key(el[t]);
                if ((kk >> sh0) == d) atomicAdd(&h[(kk >> sh1) & m2], 1u);
            }
        }
    }
    __syncthreads();
    find_threshold<Grp<NT>>(h, 1 << b2, need2, s_res, s_warp);
    const uint32_t key = (d << sh0) | (s_res[0] << sh1);
    for (int i = tid; i < (1 << b2); i += NT) h[i] = 0u;
    __syncthreads();
    return key;
}

// ---------------------------------------------------------------------------
// Exact selection over keys split into up to kMaxParts segments in column
// order (a whole row in global memory = one segment; the merged candidates of
// a split row = one segment per part, staged in shared memory or left in the
// workspace).  Single CTA.  max_tkey: the selection is valid only if every key
// of the final threshold class is >= max_tkey (each part kept only keys >= its
// own estimate); otherwise return false before anything is written.  Writes
// the k outputs (and, with GATHER, the gathered rows).
// ---------------------------------------------------------------------------
template <typename E>
struct Segments {
    int n;                                  // number of segments
    const E *bits[kMaxParts];               // raw element bits
    const int32_t *cols[kMaxParts];         // column of each element, or null: col = base + i
    int64_t base[kMaxParts];
    uint32_t pre[kMaxParts + 1];            // prefix of the segment sizes
};

template <typename E>
__device__ __forceinline__ E seg_bits(const Segments<E> &sg, int s, uint32_t i)
{
    return sg.bits[s][i];  // generic load: the segments are in shared or in global memory
}

template <typename E>
__device__ __forceinline__ int64_t seg_col(const Segments<E> &sg, int s, uint32_t i)
{
    return sg.cols[s] ? static_cast<int64_t>(__ldcg(sg.cols[s] + i)) : sg.base[s] + i;
}

template <typename E, typename G, bool GATHER>
__device__ bool select_segments(const TopkArgs &a, int64_t row, const Segments<E> &sg, uint32_t max_tkey,
                                 uint32_t *hist, uint32_t *s_res, uint32_t *s_warp, int32_t *glist)
{
    using T = Elem<E>;
    constexpr int NT = G::NT;
    const int tid = G::tid();
    const uint32_t total = sg.pre[sg.n];
    uint32_t prefix = 0, need = static_cast<uint32_t>(a.k), cnt = 0;
    int shift = T::KB;
    for (int l = 0; l < a.nlevels && (l == 0 || cnt != need); ++l) {
        const int bl = a.bits[l];
        const int nsh = shift - bl;
        const int nb = 1 << bl;
        const uint32_t mask = static_cast<uint32_t>(nb - 1);
        const int lane = tid & 31;
        for (int s = 0; s < sg.n; ++s) {
            const uint32_t cs = sg.pre[s + 1] - sg.pre[s];
            for (uint32_t b = tid & ~31u; b < cs; b += NT) {  // warp-uniform trip count
                const uint32_t i = b + lane;
                const bool in = i < cs;
                const uint32_t kk = in ? T::key(seg_bits(sg, s, i)) : 0u;
                hist_add_grouped(hist, (kk >> nsh) & mask, in && (l == 0 || (kk >> shift) == prefix), lane);
            }
        }
        G::sync();
        find_threshold<G>(hist, nb, need, s_res, s_warp);
        const uint32_t d = s_res[0];
        for (int i = tid; i < nb; i += NT) hist[i] = 0u;
        G::sync();
        if (l == 0 && d < (max_tkey >> nsh)) return false;
        prefix = (l == 0) ? d : ((prefix << bl) | d);
        need -= s_res[1];
        cnt = s_res[2];
        shift = nsh;
    }
    const uint32_t P = prefix;
    const int S = shift;
    const uint32_t E_need = need;
    if ((P << S) < max_tkey) return false;
    // ordered compaction: thread t owns the flat run [t*m, t*m + m)
    const uint32_t m = (total + NT - 1) / NT;
    const uint32_t f0 = min(total, static_cast<uint32_t>(tid) * m), f1 = min(total, f0 + m);
    int s0 = 0;
    while (s0 + 1 < sg.n && sg.pre[s0 + 1] <= f0) ++s0;
    uint32_t g = 0, q = 0;
    {
        int s = s0;
        for (uint32_t f = f0; f < f1; ++f) {
            while (f >= sg.pre[s + 1]) ++s;
            const uint32_t c = T::key(seg_bits(sg, s, f - sg.pre[s])) >> S;
            g += c > P;
            q += c == P;
        }
    }
    uint32_t tq;
    uint32_t r = block_exclusive_scan<G>(q, s_warp, tq);
    const uint32_t sel = g + take_from_ties(E_need, r, q);
    uint32_t ts;
    uint32_t pos = block_exclusive_scan<G>(sel, s_warp, ts);
    // The histogram is free now.  When it can hold a 16-bit source index per output position,
    // record which entry lands where, then write the outputs position by position: the column
    // loads are independent (many in flight) and the stores coalesce.
    const bool by_position = total <= 65535u && static_cast<uint32_t>(a.k) <= 2u * static_cast<uint32_t>(a.hist_bins);
    uint16_t *src = reinterpret_cast<uint16_t *>(hist);
    {
        int s = s0;
        for (uint32_t f = f0; f < f1; ++f) {
            while (f >= sg.pre[s + 1]) ++s;
            const uint32_t i = f - sg.pre[s];
            const E e = seg_bits(sg, s, i);
            const uint32_t c = T::key(e) >> S;
            bool take = c > P;
            if (c == P) take = (r++ < E_need);
            if (take) {
                if (by_position) {
                    if (SEL_IN_BOUNDS(pos < static_cast<uint32_t>(a.k), a.err_flag)) src[pos] = static_cast<uint16_t>(f);
                } else {
                    const int64_t col = seg_col(sg, s, i);
                    store_idx(a, row, pos, col);
                    if (a.want_values) store_val<E>(a, row, pos, e);
                    if (GATHER && static_cast<int64_t>(pos) < a.n_gather) glist[pos] = static_cast<int32_t>(col);
                }
                ++pos;
            }
        }
    }
    if (by_position) {
        G::sync();
        constexpr int U = 4;
        for (int j0 = tid; j0 < a.k; j0 += U * NT) {
            int64_t col[U];
            E val[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u * NT;
                if (j < a.k) {
                    const uint32_t f = src[j];
                    int lo = 0, hi = sg.n - 1;  // the segment holding flat index f
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (sg.pre[mid] <= f) lo = mid;
                        else hi = mid - 1;
                    }
                    const uint32_t i = f - sg.pre[lo];
                    val[u] = seg_bits(sg, lo, i);
                    col[u] = seg_col(sg, lo, i);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u * NT;
                if (j < a.k) {
                    store_idx(a, row, j, col[u]);
                    if (a.want_values) store_val<E>(a, row, j, val[u]);
                    if (GATHER && j < a.n_gather) glist[j] = static_cast<int32_t>(col[u]);
                }
            }
        }
    }
    if (GATHER) {
        G::sync();
        gather_rows_of<G>(a, row, 0, a.n_gather, glist, 0);
    }
    return true;
}

// The merged candidates of a split row after staging: segment s's keys sit in shared memory at
// byte offset stage_off[s] (16-byte aligned), the segments back to back.  Same result as
// select_segments, but every pass walks 16-byte vectors of the staged bytes (V keys at once)
// instead of single elements; the segment of a vector comes from a short binary search.
template <typename E, int NT, bool GATHER>
__device__ bool select_staged(const TopkArgs &a, int64_t row, const Segments<E> &sg, const uint32_t *stage_off,
                              uint32_t staged_bytes, const unsigned char *stage, uint32_t max_tkey, uint32_t *hist,
                              uint32_t *s_res, uint32_t *s_warp, int32_t *glist)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    const int tid = threadIdx.x, lane = tid & 31;
    const int nvec = static_cast<int>(staged_bytes >> 4);
    const uint4 *sv = reinterpret_cast<const uint4 *>(stage);
    // segment of staged vector v and the number of its keys that are real (< V in a segment's last vector)
    auto locate = [&](int v, int &seg, int &first) {
        int lo = 0, hi = sg.n - 1;
        const uint32_t byte = static_cast<uint32_t>(v) << 4;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (stage_off[mid] <= byte) lo = mid;
            else hi = mid - 1;
        }
        seg = lo;
        first = static_cast<int>((byte - stage_off[lo]) / sizeof(E));  // index of the vector's first key
        const int count = static_cast<int>(sg.pre[lo + 1] - sg.pre[lo]);
        return min(V, count - first);
    };
    uint32_t prefix = 0, need = static_cast<uint32_t>(a.k), cnt = 0;
    int shift = T::KB;
    for (int l = 0; l < a.nlevels && (l == 0 || cnt != need); ++l) {
        const int bl = a.bits[l];
        const int nsh = shift - bl;
        const int nb = 1 << bl;
        const uint32_t mask = static_cast<uint32_t>(nb - 1);
        for (int b = tid & ~31; b < nvec; b += NT) {  // warp-uniform trip count
            const int v = b + lane;
            int seg = 0, first = 0, lim = 0;
            E el[V];
            if (v < nvec) lim = locate(v, seg, first);
            T::unpack(v < nvec ? sv[v] : make_uint4(0u, 0u, 0u, 0u), el);
#pragma unroll
            for (int t = 0; t < V; ++t) {
                const uint32_t kk = T::key(el[t]);
                hist_add_grouped(hist, (kk >> nsh) & mask, t < lim && (l == 0 || (kk >> shift) == prefix), lane);
            }
        }
        __syncthreads();
        find_threshold<Grp<NT>>(hist, nb, need, s_res, s_warp);
        const uint32_t d = s_res[0];
        for (int i = tid; i < nb; i += NT) hist[i] = 0u;
        __syncthreads();
        if (l == 0 && d < (max_tkey >> nsh)) return false;
        prefix = (l == 0) ? d : ((prefix << bl) | d);
        need -= s_res[1];
        cnt = s_res[2];
        shift = nsh;
    }
    const uint32_t P = prefix;
    const int S = shift;
    const uint32_t E_need = need;
    if ((P << S) < max_tkey) return false;
    // ordered compaction over vectors: thread t owns vectors [t*m, t*m + m) (staged order = column order)
    const int m = (nvec + NT - 1) / NT;
    const int v0 = min(nvec, tid * m), v1 = min(nvec, v0 + m);
    uint32_t g = 0, q = 0;
    for (int v = v0; v < v1; ++v) {
        int seg, first;
        const int lim = locate(v, seg, first);
        E el[V];
        T::unpack(sv[v], el);
#pragma unroll
        for (int t = 0; t < V; ++t) {
            if (t < lim) {
                const uint32_t c = T::key(el[t]) >> S;
                g += c > P;
                q += c == P;
            }
        }
    }
    uint32_t tq;
    uint32_t r = block_exclusive_scan<Grp<NT>>(q, s_warp, tq);
    const uint32_t sel = g + take_from_ties(E_need, r, q);
    uint32_t ts;
    uint32_t pos = block_exclusive_scan<Grp<NT>>(sel, s_warp, ts);
    const uint32_t total = sg.pre[sg.n];
    const bool by_position = total <= 65535u && static_cast<uint32_t>(a.k) <= 2u * static_cast<uint32_t>(a.hist_bins);
    uint16_t *src = reinterpret_cast<uint16_t *>(hist);  // the histogram is free now
    for (int v = v0; v < v1; ++v) {
        int seg, first;
        const int lim = locate(v, seg, first);
        E el[V];
        T::unpack(sv[v], el);
#pragma unroll
        for (int t = 0; t < V; ++t) {
            if (t < lim) {
                const uint32_t c = T::key(el[t]) >> S;
                bool take = c > P;
                if (c == P) take = (r++ < E_need);
                if (take) {
                    const uint32_t i = static_cast<uint32_t>(first + t);
                    if (by_position) {
                        if (SEL_IN_BOUNDS(pos < static_cast<uint32_t>(a.k), a.err_flag))
                            src[pos] = static_cast<uint16_t>(sg.pre[seg] + i);
                    } else {
                        const int64_t col = seg_col(sg, seg, i);
                        store_idx(a, row, pos, col);
                        if (a.want_values) store_val<E>(a, row, pos, el[t]);
                        if (GATHER && static_cast<int64_t>(pos) < a.n_gather) glist[pos] = static_cast<int32_t>(col);
                    }
                    ++pos;
                }
            }
        }
    }
    if (by_position) {
        // output position j: its source entry, column from the workspace (independent loads), key from smem
        __syncthreads();
        constexpr int U = 4;
        for (int j0 = tid; j0 < a.k; j0 += U * NT) {
            int64_t col[U];
            E val[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u * NT;
                if (j < a.k) {
                    const uint32_t f = src[j];
                    int lo = 0, hi = sg.n - 1;
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (sg.pre[mid] <= f) lo = mid;
                        else hi = mid - 1;
                    }
                    const uint32_t i = f - sg.pre[lo];
                    val[u] = seg_bits(sg, lo, i);
                    col[u] = seg_col(sg, lo, i);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u * NT;
                if (j < a.k) {
                    store_idx(a, row, j, col[u]);
                    if (a.want_values) store_val<E>(a, row, j, val[u]);
                    if (GATHER && j < a.n_gather) glist[j] = static_cast<int32_t>(col[u]);
                }
            }
        }
    }
    if (GATHER) {
        __syncthreads();
        gather_rows_of<Grp<NT>>(a, row, 0, a.n_gather, glist, 0);
    }
    return true;
}

// ---------------------------------------------------------------------------
// reg_kernel: one CTA per row, the row held in registers.  Thread t owns a
// contiguous run of re <= R 16-byte vectors (re sized to the row's valid
// length, so short rows keep every thread busy; the part past the row's end
// is read with scalar loads, nothing beyond it), so the
// radix levels run straight from registers, and the thread order is the
// column order: one pair of block scans orders the compaction.  The
// compaction records each output position's source column in shared memory,
// and the outputs are then written in position order (coalesced).
// Shared memory: histogram | source columns (k x 16 bits) | gather list.
// ---------------------------------------------------------------------------
// Value-ordered outputs of one row (SEL_SORT_VALUE in the register and staged row kernels): the row's n_valid
// selected columns, in ascending column order, are src[0, n_valid) (src null: columns 0 ..
// n_valid-1 themselves), their values buf[col] (buf null: the row in global memory, xrow).  They
// are ranked by value (order_core.cuh; NT * 8 >= k), and output j < k gets the column of rank j
// (index -1 and the fill value past n_valid); with GATHER the first n_gather columns also go to
// glist.  `rank` is order::rank_smem_bytes of shared memory that nothing else still reads.
template <typename E, int NT, bool GATHER>
__device__ void ordered_write(const TopkArgs &a, int64_t row, int n_valid, const uint16_t *src, const E *buf,
                              const E *xrow, unsigned char *rank, int32_t *glist)
{
    using T = Elem<E>;
    constexpr bool kBf16 = sizeof(E) == 2;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int k = a.k;
    auto col_of = [&](int p) { return src ? static_cast<int>(src[p]) : p; };
    auto val_of = [&](int c) { return buf ? buf[c] : xrow[c]; };
    uint32_t v[order::kEpt];
    bool valid[order::kEpt];
#pragma unroll
    for (int e = 0; e < order::kEpt; ++e) {
        const int p = warp * order::kWarpItems + e * 32 + lane;
        valid[e] = p < n_valid;
        v[e] = valid[e] ? static_cast<uint32_t>(val_of(col_of(p))) : static_cast<uint32_t>(T::kFill);
    }
    order::value_rank<kBf16, NT>(v, valid, rank);
#pragma unroll
    for (int u = 0; u < order::kEpt; ++u) {
        const int j = t + u * NT;
        if (j >= k) break;
        const int slot = order::ranked_position<kBf16>(rank, j);
        const int c = slot < n_valid ? col_of(slot) : -1;
        store_idx(a, row, j, c);
        if (a.want_values) store_val<E>(a, row, j, c >= 0 ? val_of(c) : static_cast<E>(T::kFill));
        if (GATHER && j < a.n_gather) glist[j] = c;
    }
}

template <int NT, int R>
struct RegMinBlocks {  // a register budget that holds the run (R vectors) without spilling
    static constexpr int value = R <= 2 ? MinBlocks<NT>::value : (NT >= 512 ? 1 : (NT >= 256 ? 2 : 4));
};

template <typename E, int NT, int R, bool GATHER, bool ORDER>
__global__ void __launch_bounds__(NT, (RegMinBlocks<NT, R>::value)) reg_kernel(const TopkArgs a)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    static_assert(NT * R * V <= 65536, "source columns are 16-bit");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t s_warp[NT / 32];
    __shared__ uint32_t s_res[4];
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t row = row_of_block(a, blockIdx.x);
    const int64_t n = valid_cols(a, row);
    const int k = a.k;
    const E *xrow = static_cast<const E *>(a.x) + row * a.stride;
    if (n <= k) {
        if constexpr (ORDER) {
            int32_t *gl = GATHER ? reinterpret_cast<int32_t *>(smem + a.smem_glist_off) : nullptr;
            ordered_write<E, NT, GATHER>(a, row, static_cast<int>(n), nullptr, nullptr, xrow, smem + a.smem_order_off, gl);
            if (GATHER) {
                __syncthreads();
                gather_rows_of<Grp<NT>>(a, row, 0, a.n_gather, gl, 0);
            }
        } else {
            short_row<E, Grp<NT>, GATHER>(a, row, n, 0, k);
        }
        return;
    }
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + a.smem_hist_off);
    uint16_t *src = reinterpret_cast<uint16_t *>(smem + a.smem_list_off);
    int32_t *glist = GATHER ? reinterpret_cast<int32_t *>(smem + a.smem_glist_off) : nullptr;
    for (int i = tid; i < a.hist_bins; i += NT) hist[i] = 0u;

    // ---- the thread's run: re vectors (the row's vectors spread evenly over the threads; slots
    //      j >= re are skipped, warp-uniformly), cnt valid elements from column e0
    const int nv = static_cast<int>((n + V - 1) / V);  // vectors holding the row, the last maybe partial
    const int re = (nv + NT - 1) / NT;                 // <= R by the plan
    const int e0 = tid * re * V;
    const int cnt = static_cast<int>(n - e0 < 0 ? 0 : (n - e0 > re * V ? re * V : n - e0));
    const int nfull = cnt / V;
    const uint4 *xv = reinterpret_cast<const uint4 *>(xrow) + tid * re;
    uint4 q[R];
#pragma unroll
    for (int j = 0; j < R; ++j) q[j] = j < nfull ? __ldg(xv + j) : make_uint4(0u, 0u, 0u, 0u);
    if (nfull < re && cnt > nfull * V) {  // the row ends inside this vector: scalar loads
        E el[V];
#pragma unroll
        for (int t = 0; t < V; ++t) el[t] = nfull * V + t < cnt ? xrow[e0 + nfull * V + t] : static_cast<E>(0);
        const uint4 part = T::pack(el);
#pragma unroll
        for (int j = 0; j < R; ++j)
            if (j == nfull) q[j] = part;
    }
    uint32_t smax = T::kSmaxInit, umax = T::kUmaxInit;
#pragma unroll
    for (int j = 0; j < R; ++j)
        if (j < re) T::nan_acc(q[j], smax, umax);  // zero padding is NaN-free
    if (__syncthreads_or(T::has_nan(smax, umax)) && tid == 0 && a.nan_flag) atomicOr(a.nan_flag, 1);

    // ---- radix levels from the most significant digit, over the registers
    uint32_t prefix = 0, need = static_cast<uint32_t>(k), cls = 0;
    int shift = T::KB;
    for (int l = 0; l < a.nlevels && (l == 0 || cls != need); ++l) {
        const int bl = a.bits[l];
        const int nsh = shift - bl;
        const int nb = 1 << bl;
        const uint32_t mask = static_cast<uint32_t>(nb - 1);
        if (a.agg) {
#pragma unroll
            for (int j = 0; j < R; ++j) {
                if (j < re) {
                    E el[V];
                    T::unpack(q[j], el);
#pragma unroll
                    for (int t = 0; t < V; ++t) {
                        const uint32_t kk = T::key(el[t]);
                        hist_add_grouped(hist, (kk >> nsh) & mask,
                                         j * V + t < cnt && (l == 0 || (kk >> shift) == prefix), lane);
                    }
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < R; ++j) {
                if (j < re) {
                    E el[V];
                    T::unpack(q[j], el);
#pragma unroll
                    for (int t = 0; t < V; ++t) {
                        const uint32_t kk = T::key(el[t]);
                        if (j * V + t < cnt && (l == 0 || (kk >> shift) == prefix))
                            atomicAdd(&hist[(kk >> nsh) & mask], 1u);
                    }
                }
            }
        }
        __syncthreads();
        find_threshold<Grp<NT>>(hist, nb, need, s_res, s_warp);
        for (int i = tid; i < nb; i += NT) hist[i] = 0u;
        __syncthreads();
        prefix = (l == 0) ? s_res[0] : ((prefix << bl) | s_res[0]);
        need -= s_res[1];
        cls = s_res[2];
        shift = nsh;
    }
    const uint32_t P = prefix;
    const int S = shift;
    const uint32_t E_need = need;

    // ---- ordered compaction: the run's keys above the class, then its ties in column order
    uint32_t g = 0, qq = 0;
#pragma unroll
    for (int j = 0; j < R; ++j) {
        if (j < re) {
            E el[V];
            T::unpack(q[j], el);
#pragma unroll
            for (int t = 0; t < V; ++t) {
                const uint32_t c = T::key(el[t]) >> S;
                const bool in = j * V + t < cnt;
                g += in && c > P;
                qq += in && c == P;
            }
        }
    }
    uint32_t tq;
    uint32_t r = block_exclusive_scan<Grp<NT>>(qq, s_warp, tq);
    const uint32_t sel = g + take_from_ties(E_need, r, qq);
    uint32_t ts;
    uint32_t pos = block_exclusive_scan<Grp<NT>>(sel, s_warp, ts);
#pragma unroll
    for (int j = 0; j < R; ++j) {
        if (j < re) {
            E el[V];
            T::unpack(q[j], el);
#pragma unroll
            for (int t = 0; t < V; ++t) {
                const uint32_t c = T::key(el[t]) >> S;
                const bool in = j * V + t < cnt;
                bool take = in && c > P;
                if (in && c == P) take = r++ < E_need;
                if (take) {
                    if (SEL_IN_BOUNDS(pos < static_cast<uint32_t>(k) && e0 + j * V + t < n, a.err_flag))
                        src[pos] = static_cast<uint16_t>(e0 + j * V + t);
                    ++pos;
                }
            }
        }
    }
    __syncthreads();
    if constexpr (ORDER) {  // ranked by value (values re-read by column from L2)
        ordered_write<E, NT, GATHER>(a, row, k, src, nullptr, xrow, smem + a.smem_order_off, glist);
    } else {
        for (int p = tid; p < k; p += NT) {  // outputs in position order
            const int col = src[p];
            store_idx(a, row, p, col);
            if (a.want_values) store_val<E>(a, row, p, xrow[col]);
            if (GATHER && p < a.n_gather) glist[p] = col;
        }
    }
    if (GATHER) {
        __syncthreads();
        gather_rows_of<Grp<NT>>(a, row, 0, a.n_gather, glist, 0);
    }
}

// ---------------------------------------------------------------------------
// row_kernel: one CTA per row, the row staged whole in shared memory.
// ---------------------------------------------------------------------------
template <typename E, int NT, bool GATHER, bool ORDER>
__global__ void __launch_bounds__(NT, MinBlocks<NT>::value) row_kernel(const TopkArgs a)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    constexpr int W = NT / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t s_bar[kMaxChunks];
    __shared__ uint32_t s_warp[W];
    __shared__ uint32_t s_wgt[W], s_weq[W];
    __shared__ uint32_t s_wsel_base[W], s_weq_base[W];
    __shared__ uint32_t s_res[4];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = row_of_block(a, blockIdx.x);
    const int64_t n = valid_cols(a, row);
    const int k = a.k;
    const E *xrow = static_cast<const E *>(a.x) + row * a.stride;
    if (n <= k) {
        if constexpr (ORDER) {
            int32_t *gl = GATHER ? reinterpret_cast<int32_t *>(smem + a.smem_glist_off) : nullptr;
            ordered_write<E, NT, GATHER>(a, row, static_cast<int>(n), nullptr, nullptr, xrow, smem + a.smem_order_off, gl);
            if (GATHER) {
                __syncthreads();
                gather_rows_of<Grp<NT>>(a, row, 0, a.n_gather, gl, 0);
            }
        } else {
            short_row<E, Grp<NT>, GATHER>(a, row, n, 0, k);
        }
        return;
    }
    E *buf = reinterpret_cast<E *>(smem);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + a.smem_hist_off);
    uint8_t *masks = smem + a.smem_mask_off;
    uint16_t *list = reinterpret_cast<uint16_t *>(smem + a.smem_list_off);
    int32_t *glist = GATHER ? reinterpret_cast<int32_t *>(smem + a.smem_glist_off) : nullptr;
    const int len = static_cast<int>(n);
    const int sh0 = T::KB - a.bits[0];
    const int nb0 = 1 << a.bits[0];
    const bool sampled = a.sample_step > 1 && n >= 4LL * k && n >= static_cast<int64_t>(a.sample_min_cols);

    for (int i = tid; i < a.hist_bins; i += NT) hist[i] = 0u;
    stage_and_histogram<E, NT>(a, xrow, 0, len, sampled ? a.sample_step : 1, smem, hist, s_bar);

    // first digit: exact, or estimated from the sample and then made exact over the candidates
    int L = 0;
    bool list_ok = false;
    bool exact = false;
    if (sampled) {
        const uint32_t tkey = sample_threshold_key<E, NT>(a, buf, static_cast<int>((len * sizeof(E)) >> 4),
                                                          a.sample_step, hist, static_cast<float>(k),
                                                          static_cast<float>(n), s_res, s_warp);
        L = filter_to_list<E, NT>(a, buf, len, tkey, masks, list, a.list_cap, s_warp);
        list_ok = L <= a.list_cap;
        if (list_ok) {
            for (int b = warp * 32; b < L; b += NT) {
                const int i = b + lane;
                const bool in = i < L;
                hist_add_grouped(hist, in ? T::key(buf[list[i]]) >> sh0 : 0u, in, lane);
            }
        } else {
            const int nvt = (len + V - 1) / V;
            for (int base = warp * 32; base < nvt; base += NT) {
                const int v = base + lane;
                if (v < nvt) {
                    E el[V];
                    T::unpack(reinterpret_cast<const uint4 *>(buf)[v], el);
#pragma unroll
                    for (int t = 0; t < V; ++t) {
                        const uint32_t kk = T::key(el[t]);
                        if (v * V + t < len && kk >= tkey) atomicAdd(&hist[kk >> sh0], 1u);
                    }
                }
            }
        }
        __syncthreads();
        exact = hist_total<Grp<NT>>(hist, nb0, s_warp) >= static_cast<uint32_t>(k);
        if (!exact) {  // the estimate was too high: exact histogram of the whole slice
            for (int i = tid; i < nb0; i += NT) hist[i] = 0u;
            __syncthreads();
            const int nvt = (len + V - 1) / V;
            for (int base = warp * 32; base < nvt; base += NT) {
                const int v = base + lane;
                if (v < nvt) {
                    E el[V];
                    T::unpack(reinterpret_cast<const uint4 *>(buf)[v], el);
#pragma unroll
                    for (int t = 0; t < V; ++t)
                        if (v * V + t < len) atomicAdd(&hist[T::key(el[t]) >> sh0], 1u);
                }
            }
            __syncthreads();
        }
    }
    find_threshold<Grp<NT>>(hist, nb0, static_cast<uint32_t>(k), s_res, s_warp);
    for (int i = tid; i < nb0; i += NT) hist[i] = 0u;
    __syncthreads();
    if (!exact) {
        L = filter_to_list<E, NT>(a, buf, len, s_res[0] << sh0, masks, list, a.list_cap, s_warp);
        list_ok = L <= a.list_cap;
    }
    uint32_t prefix = s_res[0];  // selection class: (key >> shift) == prefix
    int shift = sh0;
    uint32_t need = static_cast<uint32_t>(k) - s_res[1];
    uint32_t cnt = s_res[2];
    const int nvt = (len + V - 1) / V;
    const uint4 *vbuf = reinterpret_cast<const uint4 *>(buf);

    // ---------------------------------------------------- further levels
    for (int l = 1; l < a.nlevels && cnt != need; ++l) {
        const int bl = a.bits[l];
        const int nsh = shift - bl;
        const int nb = 1 << bl;
        const uint32_t mask = static_cast<uint32_t>(nb - 1);
        if (list_ok) {
            for (int b = warp * 32; b < L; b += NT) {
                const int i = b + lane;
                const bool in = i < L;
                const uint32_t kk = in ? T::key(buf[list[i]]) : 0u;
                hist_add_grouped(hist, (kk >> nsh) & mask, in && (kk >> shift) == prefix, lane);
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
        find_threshold<Grp<NT>>(hist, nb, need, s_res, s_warp);
        for (int i = tid; i < nb; i += NT) hist[i] = 0u;
        __syncthreads();
        prefix = (prefix << bl) | s_res[0];
        need -= s_res[1];
        cnt = s_res[2];
        shift = nsh;
    }
    const uint32_t P = prefix;
    const int S = shift;
    const uint32_t E_need = need;  // keys of class P still to take, in column order

    // --------------------------------------------- ordered write of the k
    if (list_ok) {
        // thread t owns list entries [m t, m t + m); m is rounded up to 2 mod 4 so that the first
        // entries of a warp's threads (16-bit, m/2 words apart, m/2 odd) fall in distinct banks
        const int m0 = (L + NT - 1) / NT;
        const int m = m0 <= 1 ? m0 : m0 + ((6 - (m0 & 3)) & 3);
        const int i0 = min(L, tid * m), i1 = min(L, i0 + m);
        uint32_t g = 0, q = 0;
        for (int i = i0; i < i1; ++i) {
            const uint32_t c = T::key(buf[list[i]]) >> S;
            g += c > P;
            q += c == P;
        }
        uint32_t tq;
        uint32_t r = block_exclusive_scan<Grp<NT>>(q, s_warp, tq);
        const uint32_t sel = g + take_from_ties(E_need, r, q);
        uint32_t ts;
        uint32_t pos = block_exclusive_scan<Grp<NT>>(sel, s_warp, ts);
        // each output position's column goes to the (free) histogram first when it fits (16 bits
        // each); the outputs are then written in position order, coalesced
        // (value-ordered launches always fit: the plan checks k <= 2 * hist_bins)
        const bool by_position = ORDER || static_cast<uint32_t>(k) <= 2u * static_cast<uint32_t>(a.hist_bins);
        uint16_t *src = reinterpret_cast<uint16_t *>(hist);
        for (int i = i0; i < i1; ++i) {
            const int o = list[i];
            const E e = buf[o];
            const uint32_t c = T::key(e) >> S;
            bool take = c > P;
            if (c == P) take = (r++ < E_need);
            if (take) {
                if (by_position) {
                    if (SEL_IN_BOUNDS(pos < static_cast<uint32_t>(k) && pos < 2u * static_cast<uint32_t>(a.hist_bins) &&
                                          o < len,
                                      a.err_flag))
                        src[pos] = static_cast<uint16_t>(o);
                } else {
                    store_idx(a, row, pos, o);
                    if (a.want_values) store_val<E>(a, row, pos, e);
                    if (GATHER && static_cast<int64_t>(pos) < a.n_gather) glist[pos] = o;
                }
                ++pos;
            }
        }
        if (by_position) {
            __syncthreads();
            if constexpr (ORDER) {
                ordered_write<E, NT, GATHER>(a, row, k, src, buf, xrow, smem + a.smem_order_off, glist);
            } else {
                for (int p = tid; p < k; p += NT) {
                    const int o = src[p];
                    store_idx(a, row, p, o);
                    if (a.want_values) store_val<E>(a, row, p, buf[o]);
                    if (GATHER && p < a.n_gather) glist[p] = o;
                }
            }
        }
    } else {
        // full-slice path (candidates overflowed the list): warp-segment counts, then an ordered
        // write in which every warp walks its own contiguous segment
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
        if (tid == 0) {
            uint32_t ws = 0, we = 0;
            for (int w = 0; w < W; ++w) {
                s_wsel_base[w] = ws;
                s_weq_base[w] = we;
                ws += s_wgt[w] + take_from_ties(E_need, we, s_weq[w]);
                we += s_weq[w];
            }
        }
        __syncthreads();
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
                    if constexpr (ORDER) {  // the column goes to its position; ranked below
                        if (SEL_IN_BOUNDS(pos < static_cast<uint32_t>(k) && pos < 2u * static_cast<uint32_t>(a.hist_bins),
                                          a.err_flag))
                            reinterpret_cast<uint16_t *>(hist)[pos] = static_cast<uint16_t>(o + t);
                    } else {
                        store_idx(a, row, pos, o + t);
                        if (a.want_values) store_val<E>(a, row, pos, el[t]);
                        if (GATHER && static_cast<int64_t>(pos) < a.n_gather) glist[pos] = o + t;
                    }
                    ++pos;
                }
            }
            eq_run += tq;
            sel_run += ts;
        }
        if constexpr (ORDER) {
            __syncthreads();
            ordered_write<E, NT, GATHER>(a, row, k, reinterpret_cast<const uint16_t *>(hist), buf, xrow,
                                         smem + a.smem_order_off, glist);
        }
    }
    if (GATHER) {
        __syncthreads();
        gather_rows_of<Grp<NT>>(a, row, 0, a.n_gather, glist, 0);
    }
}

// ---------------------------------------------------------------------------
// split_kernel: `parts` CTAs per row; grid = rows * parts.
// Workspace (caller-owned, 256-byte aligned):
//   [0, ws_counter_bytes)         uint32 arrival counter per row (zeroed on the
//                                 stream before every launch)
//   per row r, at ws_counter_bytes + r * ws_row_bytes:
//     uint32 count[parts], uint32 tkey[parts]       (padded to 16 bytes)
//     per part p, at ws_head_bytes + p * ws_part_bytes:
//       E bits[part_cap] (padded to 16 bytes), int32 cols[part_cap]
// ---------------------------------------------------------------------------
template <typename E, int NT, bool GATHER>
__global__ void __launch_bounds__(NT, MinBlocks<NT>::value) split_kernel(const TopkArgs a)
{
    using T = Elem<E>;
    constexpr int W = NT / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint64_t s_bar[kMaxChunks];
    __shared__ uint32_t s_warp[W];
    __shared__ uint32_t s_res[4];
    __shared__ uint32_t s_last;
    __shared__ Segments<E> s_seg;
    __shared__ uint32_t s_stage_off[kMaxParts];
    __shared__ uint32_t s_staged;
    __shared__ uint64_t s_merge_bar;

    const int tid = threadIdx.x;
    const int P = a.parts;
    const int64_t row = row_of_block(a, blockIdx.x / P);
    const int part = static_cast<int>(blockIdx.x % static_cast<unsigned>(P));
    const int64_t n = valid_cols(a, row);
    const int k = a.k;
    if (n <= k) {
        if (part == 0) short_row<E, Grp<NT>, GATHER>(a, row, n, 0, k);
        return;
    }
    const E *xrow = static_cast<const E *>(a.x) + row * a.stride;
    E *buf = reinterpret_cast<E *>(smem);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + a.smem_hist_off);
    uint8_t *masks = smem + a.smem_mask_off;
    uint16_t *list = reinterpret_cast<uint16_t *>(smem + a.smem_list_off);
    int32_t *glist = GATHER ? reinterpret_cast<int32_t *>(smem + a.smem_glist_off) : nullptr;
    const int sh0 = T::KB - a.bits[0];
    const int64_t lo = static_cast<int64_t>(part) * a.slice;
    const int64_t hi = min(n, lo + a.slice);
    const int len = hi > lo ? static_cast<int>(hi - lo) : 0;

    unsigned char *wrow = a.ws + a.ws_counter_bytes + row * a.ws_row_bytes;
    if (!SEL_IN_BOUNDS(static_cast<size_t>(a.ws_counter_bytes + (row + 1) * a.ws_row_bytes) <= a.ws_bytes, a.err_flag))
        return;
    uint32_t *w_count = reinterpret_cast<uint32_t *>(wrow);
    uint32_t *w_tkey = w_count + P;
    unsigned char *wpart = wrow + a.ws_head_bytes + static_cast<int64_t>(part) * a.ws_part_bytes;
    E *w_bits = reinterpret_cast<E *>(wpart);
    int32_t *w_cols = reinterpret_cast<int32_t *>(wpart + a.ws_bits_bytes);

    // ---- local candidates: keys at or above a threshold estimated from this slice's sample
    for (int i = tid; i < a.hist_bins; i += NT) hist[i] = 0u;
    uint32_t tkey = 0;
    int L = 0;
    if (len > 0) {
        const bool sampled = len > a.list_cap && a.sample_step > 1;
        stage_and_histogram<E, NT>(a, xrow, lo, len, sampled ? a.sample_step : 1, smem, hist, s_bar);
        if (sampled) {
            // this slice's expected share of the k, plus margins
            const float share = static_cast<float>(k) * static_cast<float>(len) / static_cast<float>(n);
            tkey = sample_threshold_key<E, NT>(a, buf, static_cast<int>((len * sizeof(E)) >> 4), a.sample_step, hist,
                                               share, static_cast<float>(len), s_res, s_warp);
        }
        L = filter_to_list<E, NT>(a, buf, len, tkey, masks, list, a.list_cap, s_warp);
        const bool fits = L <= a.list_cap;
        if (fits) {
            for (int i = tid; i < L; i += NT) {
                const int o = list[i];
                if (!SEL_IN_BOUNDS(i < a.list_cap && o < len, a.err_flag)) continue;
                w_bits[i] = buf[o];
                w_cols[i] = static_cast<int32_t>(lo + o);
            }
        }
        if (tid == 0) {
            w_count[part] = fits ? static_cast<uint32_t>(L) : 0xffffffffu;
            w_tkey[part] = tkey;
        }
    } else if (tid == 0) {
        w_count[part] = 0u;
        w_tkey[part] = 0u;
    }

    // ---- arrival: the last CTA of the row to finish does the selection (its histogram must be clear)
    for (int i = tid; i < a.hist_bins; i += NT) hist[i] = 0u;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        uint32_t *counter = reinterpret_cast<uint32_t *>(a.ws) + row;
        s_last = (atomicAdd(counter, 1u) == static_cast<uint32_t>(P - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    if (tid < 32) {
        // warp 0 reads the parts' counts (lane p and p + 32) and lays out the merged segments
        const int lane = tid;
        uint32_t c[2], tk[2], bytes[2];
        bool bad = false;
        uint32_t tmax = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int p = lane + 32 * h;
            c[h] = 0u;
            tk[h] = 0u;
            if (p < P) {
                c[h] = __ldcg(w_count + p);
                tk[h] = __ldcg(w_tkey + p);
                if (c[h] == 0xffffffffu) bad = true;
            }
            tmax = max(tmax, tk[h]);
        }
        bad = __any_sync(kFull, bad);
        tmax = __reduce_max_sync(kFull, tmax);
        uint32_t pre_base = 0, off_base = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int p = lane + 32 * h;
            const uint32_t cc = bad ? 0u : c[h];
            bytes[h] = (cc * static_cast<uint32_t>(sizeof(E)) + 15u) & ~15u;
            uint32_t tot_c, tot_b;
            const uint32_t xc = warp_exclusive_scan(cc, lane, tot_c);
            const uint32_t xb = warp_exclusive_scan(bytes[h], lane, tot_b);
            if (p < P) {
                unsigned char *wp = wrow + a.ws_head_bytes + static_cast<int64_t>(p) * a.ws_part_bytes;
                s_seg.bits[p] = reinterpret_cast<const E *>(wp);
                s_seg.cols[p] = reinterpret_cast<const int32_t *>(wp + a.ws_bits_bytes);
                s_seg.base[p] = 0;
                s_seg.pre[p] = pre_base + xc;
                s_stage_off[p] = off_base + xb;
            }
            pre_base += tot_c;
            off_base += tot_b;
        }
        if (lane == 0) {
            s_seg.n = P;
            s_seg.pre[P] = pre_base;
            const bool ok = !bad && pre_base >= static_cast<uint32_t>(k);
            s_res[3] = ok ? 1u : 0u;
            s_res[2] = tmax;
            // candidate keys -> shared memory when they fit in front of the histogram
            s_staged = (ok && off_base <= a.smem_hist_off) ? off_base : 0u;
            if (s_staged) {
                fence_proxy_async_global();  // the parts' candidate stores -> the bulk copies' reads
                mbar_init(&s_merge_bar, 1);
                fence_mbar_init();
                mbar_arrive_expect_tx(&s_merge_bar, off_base);
            }
        }
        __syncwarp();
        if (s_staged) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int p = lane + 32 * h;
                if (p < P) {
                    if (bytes[h]) {
                        fence_proxy_async_global();
                        bulk_load(smem + s_stage_off[p], s_seg.bits[p], bytes[h], &s_merge_bar);
                    }
                    s_seg.bits[p] = reinterpret_cast<const E *>(smem + s_stage_off[p]);
                }
            }
        }
    }
    __syncthreads();
    if (s_staged) wait_phase(&s_merge_bar, 0u, a.err_flag);
    const bool cand_ok = s_res[3] != 0u;
    const uint32_t max_tkey = s_res[2];
    bool done = false;
    if (cand_ok) {
        done = s_staged ? select_staged<E, NT, GATHER>(a, row, s_seg, s_stage_off, s_staged, smem, max_tkey, hist,
                                                       s_res, s_warp, glist)
                        : select_segments<E, Grp<NT>, GATHER>(a, row, s_seg, max_tkey, hist, s_res, s_warp, glist);
    }
    if (!done) {
        __syncthreads();
        if (tid == 0) {
            s_seg.n = 1;
            s_seg.bits[0] = xrow;
            s_seg.cols[0] = nullptr;
            s_seg.base[0] = 0;
            s_seg.pre[0] = 0;
            s_seg.pre[1] = static_cast<uint32_t>(n);
        }
        __syncthreads();
        select_segments<E, Grp<NT>, GATHER>(a, row, s_seg, 0u, hist, s_res, s_warp, glist);
    }
}

// ---------------------------------------------------------------------------
// stream_kernel: one CTA per row; every radix pass reads the row from global
// memory.  For rows wider than the split plan covers.
// ---------------------------------------------------------------------------
template <typename E, int NT, bool GATHER>
__global__ void __launch_bounds__(NT, MinBlocks<NT>::value) stream_kernel(const TopkArgs a)
{
    using T = Elem<E>;
    constexpr int W = NT / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t s_warp[W];
    __shared__ uint32_t s_res[4];
    __shared__ Segments<E> s_seg;
    const int tid = threadIdx.x;
    const int64_t row = row_of_block(a, blockIdx.x);
    const int64_t n = valid_cols(a, row);
    if (n <= a.k) {
        short_row<E, Grp<NT>, GATHER>(a, row, n, 0, a.k);
        return;
    }
    const E *xrow = static_cast<const E *>(a.x) + row * a.stride;
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + a.smem_hist_off);
    int32_t *glist = GATHER ? reinterpret_cast<int32_t *>(smem + a.smem_glist_off) : nullptr;
    for (int i = tid; i < a.hist_bins; i += NT) hist[i] = 0u;
    uint32_t mag = 0;
    for (int64_t j = tid; j < n; j += NT) mag = max(mag, T::magnitude(xrow[j]));
    if (__syncthreads_or(mag > T::kInfMagnitude) && tid == 0 && a.nan_flag) atomicOr(a.nan_flag, 1);
    if (tid == 0) {
        s_seg.n = 1;
        s_seg.bits[0] = xrow;
        s_seg.cols[0] = nullptr;
        s_seg.base[0] = 0;
        s_seg.pre[0] = 0;
        s_seg.pre[1] = static_cast<uint32_t>(n);
    }
    __syncthreads();
    select_segments<E, Grp<NT>, GATHER>(a, row, s_seg, 0u, hist, s_res, s_warp, glist);
}

// ---------------------------------------------------------------------------
// wide_kernel: one CTA per row for rows too wide to stage whole; two CTAs
// share an SM, so one CTA's selection overlaps the other's streaming.
//  1. Threshold estimate from a sample held in registers -- the first
//     16-byte vector of every lane's stream (16 runs of 32 consecutive
//     vectors spread over the row), loaded anyway: its top-digit histogram and a
//     second digit give a key that about mu*9/8 + 3 sqrt(mu) + 4 sampled keys
//     reach (mu: the sample's share of the k).
//  2. One pass over the row, read from HBM once: warp w streams a contiguous
//     range of the row's vectors with kWideUnroll coalesced 128-bit loads in
//     flight per lane and appends the (key bits, column) pairs at or above
//     the estimate to its own region of the candidate list, in column order.
//     Each vector costs two three-way maxima and one ballot on the usual
//     (positive threshold) path; the running maxima also give the largest
//     candidate key and the NaN check.  No block-wide synchronisation while
//     streaming.
//  3. Exact selection on the regions (select_regions), using the largest
//     candidate key, tracked while streaming, to scale its digits.
//  Too few candidates, or a region overflowing, falls back to exact passes
//  over the row in global memory.
// Shared memory: histogram | candidate regions (W x region_stride pairs; the
// last pair of a region absorbs writes past its capacity) | gather list |
// staging (W x kStage 16-byte vectors, then W x kStage first columns).
// ---------------------------------------------------------------------------
constexpr int kWideUnroll = 4;
// wide_kernel: every iteration, lane 0 of a warp prefetches into L2 the warp's vectors this many
// iterations ahead (0: none), so that more of the row is on its way than the registers hold
constexpr int kWidePrefetch = 2;
constexpr int kStage = kWideStage;

// State a warp carries through the expansion of its staged vectors.
struct WideExpand {
    uint32_t off;   // pairs appended to the warp's region
    uint32_t kmax;  // largest candidate key seen by this lane (non-positive thresholds)
    bool pnan;      // a NaN among this lane's candidates (non-positive thresholds)
};

// Expands a warp's sc staged vectors (stv, with their first columns stc; one vector a lane at a time,
// in order) into (key bits, column) pairs appended to the warp's region reg at off (capacity capw;
// writes past it land on the absorbing last pair).  All 32 lanes call.
template <typename E>
__device__ __forceinline__ WideExpand wide_expand(const uint4 *stv, const int32_t *stc, int sc, uint2 *reg,
                                                  uint32_t capw, bool positive, uint32_t tsg, uint32_t tkey,
                                                  uint32_t off, uint32_t kmax, bool pnan, int lane)
{
    using T = Elem<E>;
    __syncwarp();
    for (int r0 = 0; r0 < sc; r0 += 32) {
        const int i = r0 + lane;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        int cb = 0;
        uint32_t m = 0;
        if (i < sc) {
            v = stv[i];
            cb = stc[i];
            m = positive ? T::ge_mask_raw(v, tsg) : T::ge_mask_key(v, tkey);
        }
        uint32_t tot;
        uint32_t p = off + warp_exclusive_scan(static_cast<uint32_t>(__popc(m)), lane, tot);
        while (m) {
            const int t = __ffs(m) - 1;
            m &= m - 1u;
            const E e = T::lane_of(v, t);
            if (!positive) {
                kmax = max(kmax, T::key(e));
                pnan |= T::is_nan(e);
            }
            reg[p < capw ? p : capw] = make_uint2(static_cast<uint32_t>(e), static_cast<uint32_t>(cb + t));
            ++p;
        }
        off += tot;
    }
    __syncwarp();
    return WideExpand{off, kmax, pnan};
}

// wide_expand as a call.  Measured with a memset L2 flush: the split-row variant (a part streams a
// few iterations, then merges) runs faster with the expansion out of line (bf16 [4, 204800] k=1024:
// 23.2 -> 21.2-22.8 us), the one-row-per-CTA variant slower (fp32 [256, 131072] k=4096: 46.7 ->
// 48.8 us), so only the former calls it.
template <typename E>
__device__ __noinline__ WideExpand wide_expand_call(const uint4 *stv, const int32_t *stc, int sc, uint2 *reg,
                                                    uint32_t capw, bool positive, uint32_t tsg, uint32_t tkey,
                                                    uint32_t off, uint32_t kmax, bool pnan, int lane)
{
    return wide_expand<E>(stv, stc, sc, reg, capw, positive, tsg, tkey, off, kmax, pnan, lane);
}

// Threshold key estimated from sample vectors held in registers: q[0, kSU) of each thread, those
// with bit j of `ok` set valid, `ns` valid vectors over the CTA.  share / population: the k wanted
// out of the row's n.  mu = the sample's expected share of the k; the estimate keeps
// mu*(1+1/8) + 3*sqrt(mu) + 4 sampled keys at or above it: the top digit from a histogram, a
// second digit from the sampled keys in that bin, so the key is resolved to 22 bits (fp32) or
// fully (bf16).  0 (keep everything) if that is the whole sample.  Leaves h zero.
template <typename E, int NT, int kSU, int kQ>
__device__ uint32_t estimate_threshold(const TopkArgs &a, const uint4 (&q)[kQ], uint32_t ok, int ns, float share,
                                       float population, uint32_t *h, uint32_t *s_res, uint32_t *s_warp)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    const int tid = threadIdx.x, lane = tid & 31;
    const int sh0 = T::KB - a.bits[0];
    const int nb0 = 1 << a.bits[0];
    if (a.agg) {
#pragma unroll
        for (int j = 0; j < kSU; ++j) {
            const bool okj = (ok >> j) & 1u;
            E el[V];
            T::unpack(q[j], el);
#pragma unroll
            for (int t = 0; t < V; ++t) hist_add_grouped(h, T::key(el[t]) >> sh0, okj, lane);
        }
    } else {
#pragma unroll
        for (int j = 0; j < kSU; ++j) {
            if ((ok >> j) & 1u) {
                E el[V];
                T::unpack(q[j], el);
#pragma unroll
                for (int t = 0; t < V; ++t) atomicAdd(&h[T::key(el[t]) >> sh0], 1u);
            }
        }
    }
    __syncthreads();
    const float total = static_cast<float>(ns) * V;
    const float mu = share * total / population;
    const float want = mu * 1.125f + 3.0f * sqrtf(mu) + 4.0f;
    if (want >= total) {
        for (int i = tid; i < nb0; i += NT) h[i] = 0u;
        __syncthreads();
        return 0u;
    }
    find_threshold<Grp<NT>>(h, nb0, static_cast<uint32_t>(want), s_res, s_warp);
    const uint32_t d = s_res[0];
    const uint32_t need2 = static_cast<uint32_t>(want) - s_res[1];
    for (int i = tid; i < nb0; i += NT) h[i] = 0u;
    __syncthreads();
    const int b2 = sh0 < 11 ? sh0 : 11;  // refinement digit: the next bits below the top digit
    const int sh1 = sh0 - b2;
    const uint32_t m2 = (1u << b2) - 1u;
#pragma unroll
    for (int j = 0; j < kSU; ++j) {
        if ((ok >> j) & 1u) {
            E el[V];
            T::unpack(q[j], el);
#pragma unroll
            for (int t = 0; t < V; ++t) {
                const uint32_t kk = T::key(el[t]);
                if ((kk >> sh0) == d) atomicAdd(&h[(kk >> sh1) & m2], 1u);
            }
        }
    }
    __syncthreads();
    find_threshold<Grp<NT>>(h, 1 << b2, need2, s_res, s_warp);
    const uint32_t key = (d << sh0) | (s_res[0] << sh1);
    for (int i = tid; i < (1 << b2); i += NT) h[i] = 0u;
    __syncthreads();
    return key;
}

// Exact selection over candidates kept in per-warp regions: warp w's region holds cnt[w]
// (key bits, column) pairs in column order, and the regions follow each other in column order;
// every candidate key lies in [tlo, thi].
// Fast path: one histogram level over kRangeBins digits of (key - tlo), scaled to the range
// [tlo, thi] so that the candidates spread over the bins (plain atomics); the threshold bin, if
// it holds at most kRankMax pairs, is resolved exactly by ranking its members (larger key first,
// then smaller column), and the winners are marked in place (column bit 31).  Otherwise radix
// levels over the full key find the threshold class and ballots give tie ranks.  The compaction
// then runs warp by warp over its own region (a prefix over the per-warp counts orders the
// regions), so outputs come in ascending column order.  Writes the k outputs (and, with GATHER,
// the gathered rows).  s_gq: 3 * W words of scratch; hist: hist_bins words, zero on entry
// (left dirty).
constexpr int kRangeBins = 2048;
constexpr int kRankMax = 512;

// Calls f(i, pair) for every pair i < c of a region, four pairs per lane in flight (any order).
template <typename F>
__device__ __forceinline__ void for_region(const uint2 *reg, uint32_t c, int lane, F f)
{
    uint32_t i0 = 0;
    for (; i0 + 128 <= c; i0 += 128) {
        uint2 e[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) e[u] = reg[i0 + u * 32 + lane];
#pragma unroll
        for (int u = 0; u < 4; ++u) f(i0 + u * 32 + lane, e[u]);
    }
    for (uint32_t i = i0 + lane; i < c; i += 32) f(i, reg[i]);
}

template <typename E, typename G, bool GATHER>
__device__ void select_regions(const TopkArgs &a, int64_t row, uint2 *list, int rs, const uint32_t *cnt, uint32_t tlo,
                               uint32_t thi, uint32_t *hist, uint32_t *s_res, uint32_t *s_warp, uint32_t *s_gq,
                               int32_t *glist)
{
    using T = Elem<E>;
    constexpr int NT = G::NT;
    constexpr int W = G::W;
    constexpr uint32_t kMark = 0x80000000u;
    __shared__ uint32_t s_nbin;
    const int tid = G::tid(), lane = tid & 31, warp = tid >> 5;
    uint2 *reg = list + warp * rs;
    const uint32_t c = cnt[warp];
    const uint32_t lt = (1u << lane) - 1u;
    // digit of a key in the fast path: (key - tlo) >> rsh, in [0, kRangeBins)
    const uint32_t span = thi - tlo;
    const int rsh = span < kRangeBins ? 0 : (32 - __clz(span)) - 11;
    for_region(reg, c, lane, [&](uint32_t, uint2 e) { atomicAdd(&hist[(T::key(static_cast<E>(e.x)) - tlo) >> rsh], 1u); });
    if (tid == 0) s_nbin = 0u;
    if (tid < W) s_gq[2 * W + tid] = 0u;
    G::sync();
    find_threshold<G>(hist, kRangeBins, static_cast<uint32_t>(a.k), s_res, s_warp);
    const uint32_t dstar = s_res[0], above = s_res[1], inbin = s_res[2];
    const uint32_t bneed = static_cast<uint32_t>(a.k) - above;  // taken from the threshold bin
    const bool whole = inbin == bneed;
    // kind of the compaction: 0 = range digits (the whole bin, or its marked members);
    // 1 = full-key classes (a crowded threshold bin)
    const int kind = (whole || inbin <= static_cast<uint32_t>(kRankMax)) ? 0 : 1;
    uint32_t P = 0, E_need = 0;
    int S = 0;
    if (kind == 0) {
        // per-warp counts above the bin and in it; the bin's members (key, column, list position)
        // gathered into the histogram, which is free now
        uint32_t *bk = hist, *bc = hist + kRankMax, *bi = hist + 2 * kRankMax;
        uint32_t na = 0, nin = 0;
        for_region(reg, c, lane, [&](uint32_t i, uint2 e) {
            const uint32_t kk = T::key(static_cast<E>(e.x));
            const uint32_t d = (kk - tlo) >> rsh;
            na += d > dstar;
            if (d == dstar) {
                ++nin;
                if (!whole) {
                    const uint32_t slot = atomicAdd(&s_nbin, 1u);
                    bk[slot] = kk;
                    bc[slot] = e.y;
                    bi[slot] = static_cast<uint32_t>(warp * rs) + i;
                }
            }
        });
        na = __reduce_add_sync(kFull, na);
        nin = __reduce_add_sync(kFull, nin);
        if (lane == 0) {
            s_gq[warp] = na;
            s_gq[W + warp] = nin;
        }
        G::sync();  // bin members and counts complete
        if (!whole) {
            // rank of a member among the bin's (larger key first, then smaller column): one warp
            // per member, its lanes comparing against the other members
            for (uint32_t m = warp; m < inbin; m += W) {
                const uint32_t km = bk[m], cm = bc[m];
                uint32_t beats = 0;
                for (uint32_t j = lane; j < inbin; j += 32) beats += (bk[j] > km) | ((bk[j] == km) & (bc[j] < cm));
                if (__reduce_add_sync(kFull, beats) < bneed && lane == 0) {
                    list[bi[m]].y = cm | kMark;
                    atomicAdd(&s_gq[2 * W + bi[m] / static_cast<uint32_t>(rs)], 1u);
                }
            }
            G::sync();
        }
    } else {
        for (int i = tid; i < kRangeBins; i += NT) hist[i] = 0u;
        G::sync();
        uint32_t prefix = 0, need = static_cast<uint32_t>(a.k), cls = 0;
        int shift = T::KB;
        for (int l = 0; l < a.nlevels && (l == 0 || cls != need); ++l) {
            const int bl = a.bits[l];
            const int nsh = shift - bl;
            const int nb = 1 << bl;
            const uint32_t mask = static_cast<uint32_t>(nb - 1);
            for (uint32_t i0 = 0; i0 < c; i0 += 32) {  // warp-uniform trip count
                const uint32_t i = i0 + lane;
                const bool in = i < c;
                const uint32_t kk = in ? T::key(static_cast<E>(reg[i].x)) : 0u;
                hist_add_grouped(hist, (kk >> nsh) & mask, in && (l == 0 || (kk >> shift) == prefix), lane);
            }
            G::sync();
            find_threshold<G>(hist, nb, need, s_res, s_warp);
            for (int i = tid; i < nb; i += NT) hist[i] = 0u;
            G::sync();
            prefix = (l == 0) ? s_res[0] : ((prefix << bl) | s_res[0]);
            need -= s_res[1];
            cls = s_res[2];
            shift = nsh;
        }
        P = prefix;
        S = shift;
        E_need = need;
        uint32_t g = 0, q = 0;
        for_region(reg, c, lane, [&](uint32_t, uint2 e) {
            const uint32_t cc = T::key(static_cast<E>(e.x)) >> S;
            g += cc > P;
            q += cc == P;
        });
        g = __reduce_add_sync(kFull, g);
        q = __reduce_add_sync(kFull, q);
        if (lane == 0) {
            s_gq[warp] = g;
            s_gq[W + warp] = q;
        }
        G::sync();
    }
    // outputs of the regions before this warp's (and, for full-key classes, their ties)
    auto taken_of = [&](int w, uint32_t ties_before) {
        if (kind == 1) return s_gq[w] + take_from_ties(E_need, ties_before, s_gq[W + w]);
        return s_gq[w] + (whole ? s_gq[W + w] : s_gq[2 * W + w]);
    };
    uint32_t ties = 0, pos = 0;
    for (int w = 0; w < warp; ++w) {
        pos += taken_of(w, ties);
        ties += s_gq[W + w];
    }
    // the region in order, four chunks of 32 pairs loaded ahead; output rows addressed once
    constexpr int kAhead = 4;
    int32_t *oi32 = a.out_idx && !a.idx_i64 ? static_cast<int32_t *>(a.out_idx) + row * a.out_idx_stride : nullptr;
    int64_t *oi64 = a.out_idx && a.idx_i64 ? static_cast<int64_t *>(a.out_idx) + row * a.out_idx_stride : nullptr;
    E *ov = a.want_values ? static_cast<E *>(a.out_val) + row * a.out_val_stride : nullptr;
    for (uint32_t i0 = 0; i0 < c; i0 += 32 * kAhead) {
        uint2 ev[kAhead];
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            const uint32_t i = i0 + u * 32 + lane;
            ev[u] = i < c ? reg[i] : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            const bool in = i0 + u * 32 + lane < c;
            const uint2 e = ev[u];
            const uint32_t kk = T::key(static_cast<E>(e.x));
            bool gt, eq = false;
            if (kind == 0) {
                const uint32_t d = (kk - tlo) >> rsh;
                gt = in && (d > dstar || (d == dstar && (whole || (e.y & kMark))));
            } else {
                const uint32_t cc = kk >> S;
                gt = in && cc > P;
                eq = in && cc == P;
            }
            const uint32_t be = __ballot_sync(kFull, eq);
            const bool take = gt || (eq && ties + __popc(be & lt) < E_need);
            const uint32_t bt = __ballot_sync(kFull, take);
            if (take && SEL_IN_BOUNDS(pos + __popc(bt & lt) < static_cast<uint32_t>(a.k), a.err_flag)) {
                const uint32_t p = pos + __popc(bt & lt);
                const int32_t col = static_cast<int32_t>(e.y & ~kMark);
                if (oi64) oi64[p] = col;
                else if (oi32) oi32[p] = col;
                if (ov) ov[p] = static_cast<E>(e.x);
                if (GATHER && static_cast<int64_t>(p) < a.n_gather) glist[p] = col;
            }
            ties += __popc(be);
            pos += __popc(bt);
        }
    }
    if (GATHER) {
        G::sync();
        gather_rows_of<G>(a, row, 0, a.n_gather, glist, 0);
    }
}

template <typename E, int NT, bool GATHER, bool SPLIT>
__global__ void __launch_bounds__(NT, 2) wide_kernel(const TopkArgs a)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    constexpr int W = NT / 32;
    constexpr int U = kWideUnroll;
    constexpr int kSU = kWideSampleVecsPerLane;
    static_assert(kSU <= U, "the sample comes from the first loads");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ uint32_t s_warp[W];
    __shared__ uint32_t s_res[4];
    __shared__ uint32_t s_cnt[W];
    __shared__ uint32_t s_kmax[W];
    __shared__ uint32_t s_gq[3 * W];
    __shared__ Segments<E> s_seg;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = SPLIT ? a.parts : 1;
    const int64_t row = row_of_block(a, SPLIT ? static_cast<int64_t>(blockIdx.x) / P : static_cast<int64_t>(blockIdx.x));
    const int part = SPLIT ? static_cast<int>(blockIdx.x % static_cast<unsigned>(P)) : 0;
    const int64_t n = valid_cols(a, row);
    const int k = a.k;
    if (n <= k) {
        if (part == 0) short_row<E, Grp<NT>, GATHER>(a, row, n, 0, k);
        return;
    }
    const E *xrow = static_cast<const E *>(a.x) + row * a.stride;
    const uint4 *xv = reinterpret_cast<const uint4 *>(xrow);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + a.smem_hist_off);
    uint2 *list = reinterpret_cast<uint2 *>(smem + a.smem_list_off);
    int32_t *glist = GATHER ? reinterpret_cast<int32_t *>(smem + a.smem_glist_off) : nullptr;
    const int rs = a.region_stride;
    const uint32_t capw = static_cast<uint32_t>(a.list_cap);
    const int64_t nvec = (n * static_cast<int64_t>(sizeof(E))) >> 4;  // full 16-byte vectors
    const int64_t tail0 = nvec * V;
    for (int i = tid; i < a.hist_bins; i += NT) hist[i] = 0u;

    // ---- 1. this CTA's vectors [pv0, pv1) (the row, or one of its P parts); warp w streams
    //         [vb, ve) of them, and its first loads double as the sample for the threshold
    //         estimate (kWideSampleVecsPerLane vectors per lane: 16 runs of consecutive vectors)
    const int64_t pv0 = nvec * part / P, pv1 = nvec * (part + 1) / P;
    const int64_t per = (pv1 - pv0) / W, rem = (pv1 - pv0) % W;
    const int64_t vb = pv0 + warp * per + (warp < rem ? warp : rem);
    const int64_t ve = vb + per + (warp < rem ? 1 : 0);
    uint4 q[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t v = vb + u * 32 + lane;
        q[u] = v < ve ? __ldcs(xv + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t ok = 0;
#pragma unroll
    for (int j = 0; j < kSU; ++j) ok |= static_cast<uint32_t>(vb + j * 32 + lane < ve) << j;
    int ns = 0;  // valid sample vectors over the CTA
    for (int w = 0; w < W; ++w) {
        const int64_t size = per + (w < rem ? 1 : 0);
        ns += static_cast<int>(size < 32 * kSU ? size : 32 * kSU);
    }
    __syncthreads();  // histogram cleared
    const uint32_t tkey = ns > 0 ? estimate_threshold<E, NT, kSU, U>(a, q, ok, ns, static_cast<float>(k),
                                                                     static_cast<float>(n), hist, s_res, s_warp)
                                 : 0u;

    // ---- 2. one pass: warp w streams its vectors into its region
    uint2 *reg = list + warp * rs;
    const bool positive = tkey > T::kSignKey;  // raw-bit compare suffices above +/-0
    const uint32_t tsg = tkey ^ T::kSignKey;
    uint32_t smax = T::kSmaxInit, umax = T::kUmaxInit;
    uint32_t off = 0;   // pairs appended to this warp's region (warp-uniform)
    uint32_t kmax = 0;  // largest candidate key seen by this lane (kept per key off the raw-compare path)
    // an estimate above the +inf key came from a sampled NaN
    bool pnan = tkey > T::key(static_cast<E>(T::kInfMagnitude));
    // Vectors holding a candidate are staged (16-byte vector + its first column, in column order)
    // in the warp's buffer of kStage entries, and expanded into (key, column) pairs a full
    // buffer at a time, one staged vector per lane.
    uint4 *stv = reinterpret_cast<uint4 *>(smem + a.smem_stage_off) + warp * kStage;
    int32_t *stc = reinterpret_cast<int32_t *>(smem + a.smem_stage_off + W * kStage * 16) + warp * kStage;
    int sc = 0;  // staged vectors (warp-uniform)
    auto expand = [&]() {
        const WideExpand st = SPLIT ? wide_expand_call<E>(stv, stc, sc, reg, capw, positive, tsg, tkey, off, kmax, pnan, lane)
                                    : wide_expand<E>(stv, stc, sc, reg, capw, positive, tsg, tkey, off, kmax, pnan, lane);
        off = st.off;
        kmax = st.kmax;
        pnan = st.pnan;
        sc = 0;
    };
    if (kWidePrefetch > 0 && lane == 0) {  // the first iterations' prefetches
        for (int d = 1; d < kWidePrefetch; ++d) {
            const int64_t pb = vb + static_cast<int64_t>(d) * 32 * U;
            if (pb < ve) prefetch_l2(xv + pb, static_cast<uint32_t>(min(static_cast<int64_t>(32 * U), ve - pb)) * 16u);
        }
    }
    // 32-bit vector offsets from the warp's first vector (a row holds fewer than 2^29 vectors)
    const uint4 *xw = xv + vb + lane;
    const int nvw = static_cast<int>(ve - vb);
    const int col0 = static_cast<int>(vb * V) + lane * V;  // column of this lane's vector at offset 0
    for (int off0 = 0; off0 < nvw; off0 += 32 * U) {
        if (kWidePrefetch > 0 && lane == 0) {
            const int pb = off0 + kWidePrefetch * 32 * U;
            if (pb < nvw) prefetch_l2(xw + pb, static_cast<uint32_t>(min(32 * U, nvw - pb)) * 16u);
        }
        if (off0 != 0) {
            if (off0 + 32 * U <= nvw) {  // a full iteration (warp-uniform): no bounds checks
#pragma unroll
                for (int u = 0; u < U; ++u) q[u] = __ldcs(xw + off0 + u * 32);
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = off0 + u * 32 + lane;
                    q[u] = v < nvw ? __ldcs(xw + off0 + u * 32) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            bool any;
            if (positive) {
                // zero vectors past the range select nothing and are NaN-free; the running signed /
                // unsigned maxima give the largest key and the NaN check at the end
                const uint32_t ms = T::smax_vec(q[u]);
                smax = T::smax_fold(smax, ms);
                umax = T::umax_fold(umax, q[u]);
                any = T::ge_raw(ms, tsg);
            } else {
                T::nan_acc(q[u], smax, umax);
                any = off0 + u * 32 + lane < nvw && T::ge_mask_key(q[u], tkey) != 0u;
            }
            const uint32_t b = __ballot_sync(kFull, any);
            if (b) {
                const int nb = __popc(b);
                if (sc + nb > kStage) expand();
                if (any) {
                    const int slot = sc + __popc(b & ((1u << lane) - 1u));
                    stv[slot] = q[u];
                    stc[slot] = col0 + (off0 + u * 32) * V;
                }
                sc += nb;
            }
        }
    }
    if (sc) expand();
    if (warp == W - 1 && part == P - 1) {  // the < 16-byte tail, after the last vector
        const int64_t j = tail0 + lane;
        const bool in = j < n;
        const E e = in ? xrow[j] : static_cast<E>(0);
        if (in) T::nan_acc1(e, smax, umax);
        const bool pass = in && T::key(e) >= tkey;
        const uint32_t bp = __ballot_sync(kFull, pass);
        if (pass) {
            kmax = max(kmax, T::key(e));
            const uint32_t p = off + __popc(bp & ((1u << lane) - 1u));
            reg[p < capw ? p : capw] = make_uint2(static_cast<uint32_t>(e), static_cast<uint32_t>(j));
        }
        off += __popc(bp);
    }
    if (positive) {  // the largest element, when it passes, is the largest candidate
        const uint32_t lk = T::smax_key(smax);
        kmax = max(kmax, lk >= tkey ? lk : 0u);
    }
    kmax = __reduce_max_sync(kFull, kmax);
    if (lane == 0) {
        s_cnt[warp] = off;
        s_kmax[warp] = kmax;
    }
    if (__syncthreads_or(pnan || T::has_nan(smax, umax)) && tid == 0 && a.nan_flag) atomicOr(a.nan_flag, 1);

    uint32_t tlo = tkey;  // every candidate key is at or above it
    bool over = false;    // a region (or a part's workspace) overflowed
    if constexpr (SPLIT) {
        // ---- a part: its candidates go to the workspace in column order (regions in warp order),
        //      then a header (count, estimate, largest key); the part that arrives last merges
        __shared__ uint32_t s_last;
        __shared__ uint4 s_head[kMaxParts];
        uint32_t pre = 0, tp = 0, thp = 0;
        bool povf = false;
        for (int w = 0; w < W; ++w) {
            const uint32_t c = s_cnt[w];
            pre += w < warp ? c : 0u;
            tp += c;
            povf |= c > capw;
            thp = max(thp, s_kmax[w]);
        }
        povf |= tp > static_cast<uint32_t>(a.part_cap);
        unsigned char *prow = a.ws + a.ws_counter_bytes + row * a.ws_row_bytes;
        povf |= !SEL_IN_BOUNDS(static_cast<size_t>(a.ws_counter_bytes + (row + 1) * a.ws_row_bytes) <= a.ws_bytes &&
                                   static_cast<int64_t>(P) * a.ws_part_bytes <= a.ws_row_bytes,
                               a.err_flag);
        if (!povf) {
            uint2 *dst = reinterpret_cast<uint2 *>(prow + part * a.ws_part_bytes + 16) + pre;
            const uint32_t c = s_cnt[warp];
            for (uint32_t i = lane; i < c; i += 32) __stcg(dst + i, reg[i]);
        }
        if (tid == 0)
            __stcg(reinterpret_cast<uint4 *>(prow + part * a.ws_part_bytes), make_uint4(povf ? 0xffffffffu : tp, tkey, thp, 0u));
        __threadfence();  // this thread's workspace writes, before the arrival below
        __syncthreads();
        if (tid == 0) s_last = atomicAdd(reinterpret_cast<uint32_t *>(a.ws) + row, 1u) == static_cast<uint32_t>(P - 1);
        __syncthreads();
        if (!s_last) return;
        __threadfence();  // the other parts' writes, before reading them
        if (tid < P) s_head[tid] = __ldcg(reinterpret_cast<const uint4 *>(prow + tid * a.ws_part_bytes));
        __syncthreads();
        // keys at or above the highest estimate are all in the union of the parts' lists
        uint32_t total = 0, tmax = 0, thi_all = 0;
        for (int p = 0; p < P; ++p) {
            const uint4 h = s_head[p];
            over |= h.x == 0xffffffffu;
            total += h.x == 0xffffffffu ? 0u : h.x;
            tmax = max(tmax, h.y);
            thi_all = max(thi_all, h.z);
        }
        if (!over) {
            // warp w takes the flat range [f0, f1) of the parts' lists (parts in order), keeping
            // the pairs at or above tmax in its region
            const uint32_t f0 = static_cast<uint32_t>(static_cast<uint64_t>(total) * warp / W);
            const uint32_t f1 = static_cast<uint32_t>(static_cast<uint64_t>(total) * (warp + 1) / W);
            uint32_t cw = 0, base = 0;
            int p = 0;
            while (p < P && base + s_head[p].x <= f0) base += s_head[p++].x;
            for (uint32_t f = f0; f < f1 && p < P; base += s_head[p++].x) {
                const uint32_t end = min(f1, base + s_head[p].x);
                const uint2 *pp = reinterpret_cast<const uint2 *>(prow + p * a.ws_part_bytes + 16);
                constexpr int kAhead = 4;  // chunks of 32 pairs loaded ahead
                for (uint32_t i0 = f; i0 < end; i0 += 32 * kAhead) {
                    uint2 ev[kAhead];
#pragma unroll
                    for (int u = 0; u < kAhead; ++u) {
                        const uint32_t i = i0 + u * 32 + lane;
                        ev[u] = i < end ? __ldcg(pp + (i - base)) : make_uint2(0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < kAhead; ++u) {
                        const bool keep = i0 + u * 32 + lane < end && T::key(static_cast<E>(ev[u].x)) >= tmax;
                        const uint32_t bk = __ballot_sync(kFull, keep);
                        if (keep) {
                            const uint32_t q2 = cw + __popc(bk & ((1u << lane) - 1u));
                            reg[q2 < capw ? q2 : capw] = ev[u];
                        }
                        cw += __popc(bk);
                    }
                }
                f = end;
            }
            if (lane == 0) {
                s_cnt[warp] = cw;
                s_kmax[warp] = thi_all;
            }
        }
        tlo = tmax;
        __syncthreads();
    }

    // ---- 3. exact selection on the regions, or the fallback
    uint32_t L = 0, thi = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) {
        L += s_cnt[w];
        over |= s_cnt[w] > capw;
        thi = max(thi, s_kmax[w]);
    }
    if (!over && L >= static_cast<uint32_t>(k)) {
        select_regions<E, Grp<NT>, GATHER>(a, row, list, rs, s_cnt, tlo, thi, hist, s_res, s_warp, s_gq, glist);
        return;
    }
    if (tid == 0) {
        s_seg.n = 1;
        s_seg.bits[0] = xrow;
        s_seg.cols[0] = nullptr;
        s_seg.base[0] = 0;
        s_seg.pre[0] = 0;
        s_seg.pre[1] = static_cast<uint32_t>(n);
    }
    __syncthreads();
    select_segments<E, Grp<NT>, GATHER>(a, row, s_seg, 0u, hist, s_res, s_warp, glist);
}

// ---------------------------------------------------------------------------
// flat_kernel: wide rows spread evenly over a persistent grid of one CTA per
// SM (a cooperative launch, so every CTA is resident and the bounded waits
// below on flags other CTAs publish always end).
//
// Work split.  Each row's 16-byte vectors are cut into `parts` chunks of at
// most `slice` vectors; chunk q (row q / parts, index q % parts) belongs to
// CTA q mod grid, which takes its chunks in order.  At any moment the whole
// GPU works on a band of consecutive rows, so rows finish one after another
// over the launch instead of all at its end, and every SM moves the same
// number of bytes.
//
// Streaming warps (0..23) do nothing but read and filter.  For each chunk of
// its CTA, warp w reads its 1/24 of the chunk (four coalesced 16-byte loads a
// lane in flight), tests every vector against the row's threshold estimate
// with two three-way maxima and one ballot, stages the passing vectors, and
// expands them (one ballot per element position gives every key its place)
// into its region of one of kFlatBufs chunk buffers in shared memory, in
// column order.  It then posts its count and largest key and bumps the
// buffer's completion counter.  It waits (in shared memory, bounded) only
// for the chunk's threshold and for a free buffer.
//
// Helper warps (24..31, a group on named barrier 1):
//   1. compute the threshold estimates of the rows this CTA is designated for
//      (row r: CTA r mod grid; rows needed in the first round first) from a
//      sample of 32 runs of 32 vectors spread over the row, and publish each
//      through a flag in the workspace; rows with n <= k get their fills here
//      (the streaming warps skip them);
//   2. copy each chunk's threshold from the workspace into shared memory
//      ahead of the streaming warps;
//   3. flush each finished chunk: the 24 regions, concatenated in column
//      order, go to the chunk's slot in the workspace with a header (count,
//      largest key, NaN seen), then one arrival on the row's counter; the
//      buffer is free again;
//   4. select the rows whose last chunk arrived here (select_regions over the
//      row's slots copied into shared-memory regions; a slot that overflowed,
//      or fewer than k candidates, falls back to exact passes over the row).
// A row whose last chunk is this CTA's final one is selected by all 32 warps
// together once the streaming is over, which shortens the launch's tail.
//
// Measured on fp32 [256, 131072], k = 4096: 0.15 ms against 0.055 ms for
// wide_kernel, so the automatic plan does not pick it.  The 24 streaming warps
// filter about 30 GB/s per SM (the 32 warps of two wide_kernel CTAs about 40),
// and one row's selection on the 8 helper warps takes ~16 us: copying the
// slots in from L2 and writing the outputs queue behind the streaming loads.
// The helpers fall behind and the streaming warps wait for free buffers.
//
// Workspace (caller-owned, 256-byte aligned; the first ws_counter_bytes are
// zeroed on the stream before every launch):
//   uint32 arrival counter [rows], estimate-ready flag [rows], estimate [rows]
//   per row r at ws_counter_bytes + r * ws_row_bytes, per chunk j at
//   j * ws_part_bytes: uint4 {count (or kSlotOverflow), largest key, NaN, 0},
//   uint2 pairs[part_cap]
// Shared memory: histogram (2048 words) | selection regions (flat_sel_pairs
// pairs) | staging (24 x kStage vectors, then 24 x kStage columns) | chunk
// buffers (kFlatBufs x 24 x (flat_wcap + 1) pairs).
// ---------------------------------------------------------------------------
constexpr uint32_t kSlotOverflow = 0xffffffffu;
constexpr int kFlatSW = kFlatStreamWarps;
using FlatHelp = Grp<kFlatSelWarps * 32, 1, kFlatStreamWarps * 32>;
using FlatAll = Grp<kFlatThreads, 2, 0>;

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Spins (bounded, ~2 s) until *p >= v; false on timeout.
__device__ __forceinline__ bool wait_at_least(const volatile uint32_t *p, uint32_t v)
{
    if (*p >= v) return true;
    const long long t0 = clock64();
    while (*p < v) {
        if (clock64() - t0 > kWaitCycles) return false;
        __nanosleep(64);
    }
    return true;
}

// Threshold estimate of one row from a fixed sample (32 runs of 32 consecutive vectors spread
// evenly over the row's full vectors, or all of them when fewer): the key that
// mu*(1+1/8) + 3*sqrt(mu) + 4 sampled keys reach, mu being the sample's expected share of the
// k.  Top digit from a histogram, then a second digit from the sampled keys in that bin.  0
// (keep everything) when that is the whole sample.  h: 2048 zeroed words, left zeroed.
template <typename E, typename G>
__device__ uint32_t flat_estimate(const TopkArgs &a, int64_t row, int64_t n, uint32_t *h, uint32_t *s_res,
                                  uint32_t *s_warp)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    constexpr int NT = G::NT;
    constexpr int kRuns = kFlatSampleVecs / 32;
    constexpr int PER = kFlatSampleVecs / NT;
    static_assert(kFlatSampleVecs % NT == 0, "whole loads per thread");
    const int tid = G::tid();
    const uint4 *xv = reinterpret_cast<const uint4 *>(static_cast<const E *>(a.x) + row * a.stride);
    const int64_t nv = (n * static_cast<int64_t>(sizeof(E))) >> 4;
    const int64_t m = nv < kFlatSampleVecs ? nv : kFlatSampleVecs;
    uint4 q[PER];
#pragma unroll
    for (int s = 0; s < PER; ++s) {
        const int64_t i = tid + s * NT;
        q[s] = make_uint4(0u, 0u, 0u, 0u);
        if (i < m) {
            const int64_t pos = nv <= kFlatSampleVecs ? i : (i >> 5) * (nv - 32) / (kRuns - 1) + (i & 31);
            q[s] = __ldcg(xv + pos);
        }
    }
    const int sh0 = T::KB - a.bits[0];
    const int nb0 = 1 << a.bits[0];
#pragma unroll
    for (int s = 0; s < PER; ++s) {
        if (tid + s * NT < m) {
            E el[V];
            T::unpack(q[s], el);
#pragma unroll
            for (int t = 0; t < V; ++t) atomicAdd(&h[T::key(el[t]) >> sh0], 1u);
        }
    }
    G::sync();
    const float total = static_cast<float>(m) * V;
    const float mu = static_cast<float>(a.k) * total / static_cast<float>(n);
    const float want = mu * 1.125f + 3.0f * sqrtf(mu) + 4.0f;
    if (want >= total) {
        for (int i = tid; i < nb0; i += NT) h[i] = 0u;
        G::sync();
        return 0u;
    }
    find_threshold<G>(h, nb0, static_cast<uint32_t>(want), s_res, s_warp);
    const uint32_t d = s_res[0];
    const uint32_t need2 = static_cast<uint32_t>(want) - s_res[1];
    for (int i = tid; i < nb0; i += NT) h[i] = 0u;
    G::sync();
    const int b2 = sh0 < 11 ? sh0 : 11;
    const int sh1 = sh0 - b2;
    const uint32_t m2 = (1u << b2) - 1u;
#pragma unroll
    for (int s = 0; s < PER; ++s) {
        if (tid + s * NT < m) {
            E el[V];
            T::unpack(q[s], el);
#pragma unroll
            for (int t = 0; t < V; ++t) {
                const uint32_t kk = T::key(el[t]);
                if ((kk >> sh0) == d) atomicAdd(&h[(kk >> sh1) & m2], 1u);
            }
        }
    }
    G::sync();
    find_threshold<G>(h, 1 << b2, need2, s_res, s_warp);
    const uint32_t key = (d << sh0) | (s_res[0] << sh1);
    for (int i = tid; i < (1 << b2); i += NT) h[i] = 0u;
    G::sync();
    return key;
}

// Shared state of one flat_kernel CTA.
struct FlatShared {
    uint32_t tk[kFlatQueue];          // threshold of each chunk ordinal (valid once tkseq > ordinal)
    uint32_t tkseq;                   // thresholds published for ordinals [0, tkseq)
    uint32_t bufgen[kFlatBufs];       // buffer b is free for ordinals <= bufgen[b]
    uint32_t done[kFlatBufs];         // streaming warps finished with buffer b (cumulative)
    uint32_t wcnt[kFlatBufs][kFlatStreamWarps];  // per buffer and warp: pairs kept (or kSlotOverflow)
    uint32_t wmax[kFlatBufs][kFlatStreamWarps];  // largest key kept
    uint32_t wnan[kFlatBufs][kFlatStreamWarps];  // NaN seen
    uint32_t defer;                   // row + 1 left for the whole CTA to select (0: none)
    uint32_t item;                    // broadcast within the helper group
    uint32_t s_warp[32], s_res[4], s_cnt[32], s_gq[96], s_pre[kFlatMaxParts + 2];
};

// The streaming warps' side (see above).
template <typename E>
__device__ void flat_stream(const TopkArgs &a, unsigned char *smem, FlatShared &fs)
{
    using T = Elem<E>;
    constexpr int V = T::V;
    constexpr int U = kWideUnroll;
    constexpr int SW = kFlatSW;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    const int64_t G = gridDim.x;
    const int cpr = a.parts;
    const int64_t nchunks = a.rows * cpr;
    const int64_t nvr = (a.cols * static_cast<int64_t>(sizeof(E))) >> 4;  // full vectors of a whole row
    const uint32_t wcap = static_cast<uint32_t>(a.flat_wcap);
    uint4 *stv = reinterpret_cast<uint4 *>(smem + a.smem_stage_off) + warp * kStage;
    int32_t *stc = reinterpret_cast<int32_t *>(smem + a.smem_stage_off + SW * kStage * 16) + warp * kStage;
    volatile uint32_t *vtkseq = &fs.tkseq;
    int ci = 0;
    for (int64_t q = blockIdx.x; q < nchunks; q += G, ++ci) {
        const int64_t row = q / cpr;
        const int j = static_cast<int>(q - row * cpr);
        const int64_t n = valid_cols(a, row);
        if (n <= a.k) continue;  // short row: its designated CTA writes the fills
        const int64_t nv = (n * static_cast<int64_t>(sizeof(E))) >> 4;
        const int64_t c0 = min(static_cast<int64_t>(j) * a.slice, nv);
        const int64_t c1 = min(min((static_cast<int64_t>(j) + 1) * a.slice, nvr), nv);
        const int64_t len = c1 - c0, per = len / SW, rem = len % SW;
        const int64_t vb = c0 + warp * per + min(static_cast<int64_t>(warp), rem);
        const int64_t ve = vb + per + (warp < rem ? 1 : 0);
        const bool has_tail = j == cpr - 1 && warp == SW - 1 && nv * V < n;
        const E *xrow = static_cast<const E *>(a.x) + row * a.stride;
        const uint4 *xv = reinterpret_cast<const uint4 *>(xrow);
        const int b = ci % kFlatBufs;
        uint2 *reg = reinterpret_cast<uint2 *>(smem + a.smem_cbuf_off) + (b * SW + warp) * (wcap + 1);
        // the first loads go out before the waits
        uint4 q4[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = vb + u * 32 + lane;
            q4[u] = v < ve ? __ldcs(xv + v) : make_uint4(0u, 0u, 0u, 0u);
        }
        bool ok = wait_at_least(vtkseq, static_cast<uint32_t>(ci) + 1u);
        ok = wait_at_least(&fs.bufgen[b], static_cast<uint32_t>(ci)) && ok;
        if (!ok) set_err(a.err_flag, kStatusTimeout);
        const uint32_t tkey = static_cast<volatile uint32_t *>(fs.tk)[ci];
        const bool positive = tkey > T::kSignKey;  // raw-bit compares suffice above +/-0
        const uint32_t tsg = tkey ^ T::kSignKey;
        uint32_t smax = T::kSmaxInit, umax = T::kUmaxInit, kmax = 0, off = 0;
        int sc = 0;
        auto expand = [&]() {
            __syncwarp();
            for (int r0 = 0; r0 < sc; r0 += 32) {
                const int i = r0 + lane;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                int cb = 0;
                uint32_t m = 0;
                if (i < sc) {
                    v = stv[i];
                    cb = stc[i];
                    m = positive ? T::ge_mask_raw(v, tsg) : T::ge_mask_key(v, tkey);
                }
                uint32_t before = 0, tot = 0;
#pragma unroll
                for (int t = 0; t < V; ++t) {
                    const uint32_t bt = __ballot_sync(kFull, (m >> t) & 1u);
                    before += __popc(bt & lt);
                    tot += __popc(bt);
                }
                uint32_t p = off + before;
#pragma unroll
                for (int t = 0; t < V; ++t) {
                    if ((m >> t) & 1u) {
                        const E e = T::lane_of(v, t);
                        if (!positive) kmax = max(kmax, T::key(e));
                        reg[p < wcap ? p : wcap] = make_uint2(static_cast<uint32_t>(e), static_cast<uint32_t>(cb + t));
                        ++p;
                    }
                }
                off += tot;
            }
            sc = 0;
            __syncwarp();
        };
        for (int64_t base = vb; base < ve; base += 32 * U) {
            if (base != vb) {
                if (base + 32 * U <= ve) {
#pragma unroll
                    for (int u = 0; u < U; ++u) q4[u] = __ldcs(xv + base + u * 32 + lane);
                } else {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int64_t v = base + u * 32 + lane;
                        q4[u] = v < ve ? __ldcs(xv + v) : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                bool any;
                if (positive) {
                    // zero vectors past the range pass nothing and hold no NaN
                    const uint32_t ms = T::smax_vec(q4[u]);
                    smax = T::smax_fold(smax, ms);
                    umax = T::umax_fold(umax, q4[u]);
                    any = T::ge_raw(ms, tsg);
                } else {
                    T::nan_acc(q4[u], smax, umax);
                    any = base + u * 32 + lane < ve && T::ge_mask_key(q4[u], tkey) != 0u;
                }
                const uint32_t bb = __ballot_sync(kFull, any);
                if (bb) {
                    const int nb = __popc(bb);
                    if (sc + nb > kStage) expand();
                    if (any) {
                        const int slot = sc + __popc(bb & lt);
                        stv[slot] = q4[u];
                        stc[slot] = static_cast<int32_t>((base + u * 32 + lane) * V);
                    }
                    sc += nb;
                }
            }
        }
        if (sc) expand();
        if (has_tail) {
            const int64_t jt = nv * V + lane;
            const bool in = jt < n;
            const E e = in ? xrow[jt] : static_cast<E>(0);
            if (in) T::nan_acc1(e, smax, umax);
            const bool pass = in && T::key(e) >= tkey;
            const uint32_t bp = __ballot_sync(kFull, pass);
            if (pass) {
                kmax = max(kmax, T::key(e));
                const uint32_t p = off + __popc(bp & lt);
                reg[p < wcap ? p : wcap] = make_uint2(static_cast<uint32_t>(e), static_cast<uint32_t>(jt));
            }
            off += __popc(bp);
        }
        // on the raw-compare path the largest candidate is the largest element when it passes
        if (positive) {
            const uint32_t lk = T::smax_key(smax);
            kmax = max(kmax, lk >= tkey ? lk : 0u);
        }
        kmax = __reduce_max_sync(kFull, kmax);
        const bool nan = __any_sync(kFull, T::has_nan(smax, umax));
        if (lane == 0) {
            fs.wcnt[b][warp] = off > wcap ? kSlotOverflow : off;
            fs.wmax[b][warp] = kmax;
            fs.wnan[b][warp] = nan ? 1u : 0u;
            __threadfence_block();
            atomicAdd(&fs.done[b], 1u);
        }
        __syncwarp();
    }
}

// Selection of one row whose chunk slots are all in the workspace, by the warp group G
// (select_regions over the slots copied into shared-memory regions, or the exact fallback).
// hist: 2048 words, zeroed on entry and on exit.
template <typename E, typename G>
__device__ void flat_select_row(const TopkArgs &a, int64_t row, unsigned char *smem, FlatShared &fs,
                                Segments<E> &s_seg)
{
    constexpr int NT = G::NT, W = G::W;
    __shared__ uint32_t s_ok, s_thi;
    const int gt = G::tid(), lane = gt & 31, gw = gt >> 5;
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + a.smem_hist_off);
    uint2 *list = reinterpret_cast<uint2 *>(smem + a.smem_list_off);
    const int rs = (a.flat_sel_pairs / W) & ~1;
    const uint32_t capw = static_cast<uint32_t>(rs - 1);
    const uint32_t *tkeys = reinterpret_cast<const uint32_t *>(a.ws) + 2 * a.rows;
    const unsigned char *wrow = a.ws + a.ws_counter_bytes + row * a.ws_row_bytes;
    const int cpr = a.parts;
    // the slots' counts (one per chunk) -> prefix in s_pre
    if (gt < 32) {
        uint32_t c = 0, thi = 0;
        bool bad = false;
        uint32_t run = 0;
        for (int s0 = 0; s0 < cpr; s0 += 32) {
            const int s = s0 + gt;
            uint4 h = make_uint4(0u, 0u, 0u, 0u);
            if (s < cpr) {
                if (SEL_IN_BOUNDS(static_cast<size_t>(a.ws_counter_bytes + row * a.ws_row_bytes + (s + 1) * a.ws_part_bytes) <=
                                      a.ws_bytes,
                                  a.err_flag))
                    h = __ldcg(reinterpret_cast<const uint4 *>(wrow + static_cast<int64_t>(s) * a.ws_part_bytes));
                else
                    h.x = kSlotOverflow;
            }
            bad |= h.x == kSlotOverflow;
            c = h.x == kSlotOverflow ? 0u : h.x;
            thi = max(thi, h.y);
            uint32_t tot;
            const uint32_t ex = warp_exclusive_scan(c, lane, tot);
            if (s < cpr) fs.s_pre[s] = run + ex;
            run += tot;
        }
        thi = __reduce_max_sync(kFull, thi);
        bad = __any_sync(kFull, bad);
        if (gt == 0) {
            fs.s_pre[cpr] = run;
            s_thi = thi;
            s_ok = (!bad && run >= static_cast<uint32_t>(a.k) && run <= static_cast<uint32_t>(W) * capw) ? 1u : 0u;
        }
    }
    G::sync();
    const uint32_t total = fs.s_pre[cpr];
    if (s_ok) {
        // warp gw copies the flat range [f0, f1) of the slots (in column order) into its region
        const uint32_t f0 = static_cast<uint32_t>(static_cast<uint64_t>(total) * gw / W);
        const uint32_t f1 = static_cast<uint32_t>(static_cast<uint64_t>(total) * (gw + 1) / W);
        uint2 *reg = list + gw * rs;
        int s = 0;
        while (s < cpr - 1 && fs.s_pre[s + 1] <= f0) ++s;
        for (uint32_t f = f0; f < f1;) {
            while (s < cpr - 1 && fs.s_pre[s + 1] <= f) ++s;
            const uint32_t end = min(f1, fs.s_pre[s + 1]);
            const uint2 *sp =
                reinterpret_cast<const uint2 *>(wrow + static_cast<int64_t>(s) * a.ws_part_bytes + 16) - fs.s_pre[s];
            uint32_t i = f + lane;
            for (; i + 96 < end; i += 128) {
                const uint2 e0 = __ldcg(sp + i), e1 = __ldcg(sp + i + 32), e2 = __ldcg(sp + i + 64),
                            e3 = __ldcg(sp + i + 96);
                reg[i - f0] = e0;
                reg[i + 32 - f0] = e1;
                reg[i + 64 - f0] = e2;
                reg[i + 96 - f0] = e3;
            }
            for (; i < end; i += 32) reg[i - f0] = __ldcg(sp + i);
            f = end;
        }
        if (lane == 0) fs.s_cnt[gw] = f1 - f0;
        G::sync();
        select_regions<E, G, false>(a, row, list, rs, fs.s_cnt, __ldcg(tkeys + row), s_thi, hist, fs.s_res,
                                    fs.s_warp, fs.s_gq, nullptr);
    } else {
        if (gt == 0) {
            s_seg.n = 1;
            s_seg.bits[0] = static_cast<const E *>(a.x) + row * a.stride;
            s_seg.cols[0] = nullptr;
            s_seg.base[0] = 0;
            s_seg.pre[0] = 0;
            s_seg.pre[1] = static_cast<uint32_t>(valid_cols(a, row));
        }
        G::sync();
        select_segments<E, G, false>(a, row, s_seg, 0u, hist, fs.s_res, fs.s_warp, nullptr);
    }
    G::sync();
    for (int i = gt; i < a.hist_bins; i += NT) hist[i] = 0u;
    G::sync();
}

// The helper warps' side (see above).  Leaves in fs.defer the row (+ 1) for the whole CTA.
template <typename E>
__device__ void flat_help(const TopkArgs &a, unsigned char *smem, FlatShared &fs, Segments<E> &s_seg)
{
    using S = FlatHelp;
    constexpr int NT = S::NT, SW = kFlatSW;
    const int gt = S::tid(), lane = gt & 31;
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + a.smem_hist_off);
    uint32_t *ctr = reinterpret_cast<uint32_t *>(a.ws);
    uint32_t *flag = ctr + a.rows;
    uint32_t *tkeys = flag + a.rows;
    const int64_t G = gridDim.x;
    const int cpr = a.parts;
    const int64_t nchunks = a.rows * cpr;
    const int nci = blockIdx.x < nchunks ? static_cast<int>((nchunks - 1 - blockIdx.x) / G) + 1 : 0;
    const uint32_t wcap = static_cast<uint32_t>(a.flat_wcap);
    volatile uint32_t *vtkseq = &fs.tkseq;
    for (int i = gt; i < a.hist_bins; i += NT) hist[i] = 0u;
    // the first chunk's rows are prefetched into L2 while the estimates are worked out
    if (nci > 0) {
        const int64_t row = blockIdx.x / cpr;
        const int j = static_cast<int>(blockIdx.x - row * cpr);
        const int64_t n = valid_cols(a, row);
        const int64_t nv = n > a.k ? (n * static_cast<int64_t>(sizeof(E))) >> 4 : 0;  // inside [0, n) only
        const int64_t c0 = static_cast<int64_t>(j) * a.slice, c1 = min(c0 + a.slice, nv);
        const unsigned char *base = reinterpret_cast<const unsigned char *>(static_cast<const E *>(a.x) + row * a.stride);
        for (int64_t v = c0 + static_cast<int64_t>(gt) * 64; v < c1; v += static_cast<int64_t>(NT) * 64)
            prefetch_l2(base + v * 16, static_cast<uint32_t>(min(static_cast<int64_t>(64), c1 - v) * 16));
    }
    S::sync();
    // ---- 1. designated rows: short-row fills or the threshold estimate; rows needed in the
    //         first round (r * cpr < grid) first
    auto designated = [&](bool first_round) {
        for (int64_t r = blockIdx.x; r < a.rows; r += G) {
            if ((r * cpr < G) != first_round) continue;
            const int64_t n = valid_cols(a, r);
            if (n <= a.k) {
                short_row<E, S, false>(a, r, n, 0, a.k);
                continue;
            }
            const uint32_t t = flat_estimate<E, S>(a, r, n, hist, fs.s_res, fs.s_warp);
            if (gt == 0) {
                tkeys[r] = t;
                __threadfence();
                st_release_gpu(flag + r, 1u);
            }
        }
    };
    // copies the thresholds of this CTA's chunks whose row estimate is out, in order; `block`:
    // wait (bounded) for the next one
    auto publish = [&](bool block) {
        if (gt == 0) {
            uint32_t s = *vtkseq;
            while (static_cast<int>(s) < nci) {
                const int64_t row = (blockIdx.x + static_cast<int64_t>(s) * G) / cpr;
                uint32_t t = 0;
                if (valid_cols(a, row) > a.k) {
                    if (ld_acquire_gpu(flag + row) == 0u) {
                        if (!block) break;
                        const long long t0 = clock64();
                        bool ok = true;
                        while (ld_acquire_gpu(flag + row) == 0u) {
                            if (clock64() - t0 > kWaitCycles) {
                                ok = false;
                                break;
                            }
                            __nanosleep(128);
                        }
                        if (!ok) {
                            set_err(a.err_flag, kStatusTimeout);  // the streaming warps go on with key 0
                        }
                    }
                    t = __ldcg(tkeys + row);
                }
                fs.tk[s] = t;
                __threadfence_block();
                *vtkseq = ++s;
                block = false;
            }
        }
    };
    designated(true);
    publish(true);
    designated(false);
    // ---- 2./3./4. the chunk loop
    uint32_t expect[kFlatBufs] = {};
    int64_t defer = -1;
    for (int ci = 0; ci < nci; ++ci) {
        publish(static_cast<int>(*vtkseq) <= ci + 1);  // keep two thresholds ahead
        const int64_t q = blockIdx.x + static_cast<int64_t>(ci) * G;
        const int64_t row = q / cpr;
        const int j = static_cast<int>(q - row * cpr);
        const int b = ci % kFlatBufs;
        if (valid_cols(a, row) <= a.k) {  // short row: nothing streamed, nothing flushed
            if (gt == 0) {
                __threadfence_block();
                atomicMax(&fs.bufgen[b], static_cast<uint32_t>(ci + kFlatBufs));
            }
            continue;
        }
        expect[b] += SW;
        if (gt == 0 && !wait_at_least(&fs.done[b], expect[b])) set_err(a.err_flag, kStatusTimeout);
        S::sync();
        // flush: the 24 regions, concatenated, into the chunk's slot
        unsigned char *slot = a.ws + a.ws_counter_bytes + row * a.ws_row_bytes + static_cast<int64_t>(j) * a.ws_part_bytes;
        const bool slot_ok =
            SEL_IN_BOUNDS(static_cast<size_t>(a.ws_counter_bytes + row * a.ws_row_bytes + (j + 1) * a.ws_part_bytes) <=
                              a.ws_bytes &&
                              16 + static_cast<int64_t>(SW) * wcap * 8 <= a.ws_part_bytes,
                          a.err_flag);
        uint2 *dst = reinterpret_cast<uint2 *>(slot + 16);
        const uint2 *src = reinterpret_cast<const uint2 *>(smem + a.smem_cbuf_off) + b * SW * (wcap + 1);
        if (gt < 32) {
            const volatile uint32_t *vcnt = fs.wcnt[b], *vmax = fs.wmax[b], *vnan = fs.wnan[b];
            const uint32_t c = lane < SW ? vcnt[lane] : 0u;
            const bool ovf = __any_sync(kFull, c == kSlotOverflow);
            uint32_t tot;
            const uint32_t ex = warp_exclusive_scan(ovf ? 0u : c, lane, tot);
            if (lane < SW) fs.s_pre[lane] = slot_ok ? ex : 0u;
            const uint32_t km = __reduce_max_sync(kFull, lane < SW ? vmax[lane] : 0u);
            const bool nan = __any_sync(kFull, lane < SW && vnan[lane] != 0u);
            if (lane == 0) {
                fs.s_pre[SW] = ovf || !slot_ok ? 0u : tot;
                if (slot_ok)
                    __stcg(reinterpret_cast<uint4 *>(slot), make_uint4(ovf ? kSlotOverflow : tot, km, nan ? 1u : 0u, 0u));
                if (nan && a.nan_flag) atomicOr(a.nan_flag, 1);
            }
        }
        S::sync();
        {
            // warp w' of the group copies regions w', w' + 8, ... (each a contiguous run of the slot)
            for (int w = gt >> 5; w < SW; w += S::W) {
                const uint32_t p0 = fs.s_pre[w], cnt = fs.s_pre[w + 1] - p0;
                const uint2 *srcw = src + w * (wcap + 1);
                for (uint32_t i = lane; i < cnt; i += 32) __stcg(dst + p0 + i, srcw[i]);
            }
        }
        S::sync();
        if (gt == 0) {
            __threadfence();  // the slot, before the arrival
            const bool last = atomicAdd(ctr + row, 1u) == static_cast<uint32_t>(cpr - 1);
            fs.item = last ? static_cast<uint32_t>(row) + 1u : 0u;
            __threadfence_block();
            atomicMax(&fs.bufgen[b], static_cast<uint32_t>(ci + kFlatBufs));  // the buffer is free
        }
        S::sync();
        const uint32_t item = fs.item;
        S::sync();
        if (item) {
            __threadfence();  // the other chunks' slots (their arrivals came before ours)
            if (ci == nci - 1)
                defer = static_cast<int64_t>(item) - 1;  // this CTA's last chunk: all warps select it
            else
                flat_select_row<E, S>(a, static_cast<int64_t>(item) - 1, smem, fs, s_seg);
        }
    }
    if (gt == 0) fs.defer = static_cast<uint32_t>(defer + 1);
}

template <typename E, bool GATHER>
__global__ void __launch_bounds__(kFlatThreads, 1) flat_kernel(const TopkArgs a)
{
    static_assert(!GATHER, "flat_kernel has no fused gather");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ FlatShared fs;
    __shared__ Segments<E> s_seg;
    for (int i = threadIdx.x; i < kFlatQueue; i += blockDim.x) fs.tk[i] = 0u;
    if (threadIdx.x < kFlatBufs) {
        fs.bufgen[threadIdx.x] = threadIdx.x;
        fs.done[threadIdx.x] = 0u;
    }
    if (threadIdx.x == 0) {
        fs.tkseq = 0u;
        fs.defer = 0u;
    }
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < kFlatSW * 32)
        flat_stream<E>(a, smem, fs);
    else
        flat_help<E>(a, smem, fs, s_seg);
    // the row (if any) whose last chunk was this CTA's final one: selected by every warp
    FlatAll::sync();
    const uint32_t d = fs.defer;
    if (d) flat_select_row<E, FlatAll>(a, static_cast<int64_t>(d) - 1, smem, fs, s_seg);
}

// Self-test of the bounded wait above: one thread arms an mbarrier for 16 bytes that no copy will
// ever deliver (none is issued), and every thread waits on it with a budget of `cycles`.  The
// wait runs out, records SEL_ETIMEOUT in err_flag, and the CTA returns with nothing in flight.
__global__ void wait_selftest_kernel(int32_t *err_flag, long long cycles)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar, 16);
    }
    __syncthreads();
    wait_phase(&bar, 0u, err_flag, cycles);
}

// Raises a kernel's dynamic shared-memory limit once per device; later calls that need no more
// than what was set skip the driver call.
template <typename K>
cudaError_t raise_smem_limit(K kern, int *set_smem, size_t smem)
{
    constexpr int kMaxDevices = 64;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    if (!cacheable || set_smem[dev] < static_cast<int>(smem)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (cacheable) set_smem[dev] = static_cast<int>(smem);
    }
    return cudaSuccess;
}

// Kernel of a mode for one element type, CTA size and gather flag; null where that combination
// is never launched (row_kernel, its value-ordered variant and reg_kernel with 8 vectors a
// thread: 128/256/512 threads;
// reg_kernel with 2 vectors a thread: 128; split_kernel: 256; stream and wide: 512).
template <typename E, int NT, bool G>
void (*kernel_of(int mode))(TopkArgs)
{
    if constexpr (NT <= 512) {
        if (mode == kModeRow) return row_kernel<E, NT, G, false>;
        if (mode == kModeRowOrdered) return row_kernel<E, NT, G, true>;
        if (mode == kModeReg8) return reg_kernel<E, NT, 8, G, false>;
        if (mode == kModeReg8Ordered) return reg_kernel<E, NT, 8, G, true>;
    }
    if constexpr (NT == 128) {
        if (mode == kModeReg2) return reg_kernel<E, NT, 2, G, false>;
        if (mode == kModeReg2Ordered) return reg_kernel<E, NT, 2, G, true>;
    }
    if constexpr (NT == 256) {
        if (mode == kModeSplit) return split_kernel<E, NT, G>;
    }
    if constexpr (NT == 512) {
        if (mode == kModeStream) return stream_kernel<E, NT, G>;
        if (mode == kModeWide) return wide_kernel<E, NT, G, false>;
        if (mode == kModeWideSplit) return wide_kernel<E, NT, G, true>;
    }
    if constexpr (NT == kFlatThreads && !G) {
        if (mode == kModeFlat) return flat_kernel<E, false>;
    }
    return nullptr;
}

template <typename E, int NT, bool G>
cudaError_t launch_one(int mode, size_t smem, const TopkArgs &a, cudaStream_t stream, int64_t grid, bool query,
                       int *blocks_per_sm)
{
    static int set_smem[kNumModes][64] = {};
    void (*kern)(TopkArgs) = kernel_of<E, NT, G>(mode);
    if (!kern || mode < 0 || mode >= kNumModes) return cudaErrorInvalidValue;
    cudaError_t e = raise_smem_limit(kern, set_smem[mode], smem);
    if (e != cudaSuccess) return e;
    if (query) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, kern, NT, smem);
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (mode == kModeFlat) {
        // every CTA must be resident: the streaming warps wait on flags other CTAs publish
        void *args[] = {const_cast<TopkArgs *>(&a)};
        return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(static_cast<unsigned>(grid)),
                                           dim3(NT), args, smem, stream);
    }
    kern<<<dim3(static_cast<unsigned>(grid)), dim3(NT), smem, stream>>>(a);
    return cudaGetLastError();
}

// Dispatch over (threads, gather) for one element type.  Thread counts: row_kernel 128/256/512,
// split_kernel 256, stream_kernel and wide_kernel 512.
template <typename E>
cudaError_t launch_e(int mode, int threads, bool gather, size_t smem, const TopkArgs &a, cudaStream_t s,
                     int64_t grid, bool query, int *blocks_per_sm)
{
    if (mode == kModeSplit) {
        if (threads != 256) return cudaErrorInvalidValue;
        return gather ? launch_one<E, 256, true>(mode, smem, a, s, grid, query, blocks_per_sm)
                      : launch_one<E, 256, false>(mode, smem, a, s, grid, query, blocks_per_sm);
    }
    if (mode == kModeFlat) {
        if (threads != kFlatThreads || gather) return cudaErrorInvalidValue;
        return launch_one<E, kFlatThreads, false>(mode, smem, a, s, grid, query, blocks_per_sm);
    }
    if (mode == kModeStream || mode == kModeWide || mode == kModeWideSplit) {
        if (threads != 512) return cudaErrorInvalidValue;
        return gather ? launch_one<E, 512, true>(mode, smem, a, s, grid, query, blocks_per_sm)
                      : launch_one<E, 512, false>(mode, smem, a, s, grid, query, blocks_per_sm);
    }
    switch (threads) {
    case 128:
        return gather ? launch_one<E, 128, true>(mode, smem, a, s, grid, query, blocks_per_sm)
                      : launch_one<E, 128, false>(mode, smem, a, s, grid, query, blocks_per_sm);
    case 256:
        return gather ? launch_one<E, 256, true>(mode, smem, a, s, grid, query, blocks_per_sm)
                      : launch_one<E, 256, false>(mode, smem, a, s, grid, query, blocks_per_sm);
    case 512:
        return gather ? launch_one<E, 512, true>(mode, smem, a, s, grid, query, blocks_per_sm)
                      : launch_one<E, 512, false>(mode, smem, a, s, grid, query, blocks_per_sm);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace sel
