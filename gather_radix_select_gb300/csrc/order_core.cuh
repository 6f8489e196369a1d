// order_core.cuh -- value ranking of one row's selected entries inside a CTA.
//
// "Speed up PyTorch TopK with DeepSelect", "Performance and advanced tips"
// (item 3): results may be ordered by value.  A row's selected entries arrive
// in ascending column order; ranking them by value with a STABLE sort then
// gives equal values in column order.  The sort is a least-significant-digit
// radix sort on each value's inverted order-preserving key (-0 folded onto +0,
// any NaN above every number), rebased to the row's smallest key so that only
// the bits in which the keys differ are sorted; entries without a column
// (fills) take the key one above the range and so stay last.
//
// Each pass ranks 8-bit digits: a warp finds the lanes holding equal digits in
// each of its item rows (with one ballot per digit bit, or with match on rows
// of few distinct digits), the lowest lane of each
// group advances the warp's counter for the digit, one block-wide exclusive
// scan turns the per-warp counts into digit-major, warp-minor bases (stable),
// and each item is scattered to its rank.  Items sit warp-striped: item e of
// lane l in warp w is position 256 w + 32 e + l, so positions and the ranking
// order agree.  Every item carries its position (12 bits) below the key.
//
// Shared by the ordering kernel (order.cu) and the staged row kernel's
// value-ordered variant (topk_impl.cuh).
#pragma once

#include <cstdint>
#include <type_traits>

namespace sel {
namespace order {

constexpr int kEpt = 8;        // items a thread holds
constexpr int kSlotBits = 12;  // positions < 4096
constexpr int kRadixBits = 8;
constexpr int kDigits = 1 << kRadixBits;
constexpr int kWarpItems = 32 * kEpt;
constexpr int kBallotOnlyBits = 4;    // digits this narrow always take ballots
constexpr int kMatchMaxDistinct = 16; // a warp's first row with at most this many digits: match

// Item word: 32 bits suffice for bf16 keys (17 bits with the fill) and the 12-bit position.
template <bool BF16>
using Item = typename std::conditional<BF16, uint32_t, uint64_t>::type;

// Shared bytes value_rank needs for NT threads (items, per-warp digit counters, digit bases).
template <bool BF16>
__host__ __device__ constexpr size_t rank_smem_bytes(int nt)
{
    return static_cast<size_t>(nt) * kEpt * sizeof(Item<BF16>) +
           (static_cast<size_t>(nt / 32) * kDigits + kDigits) * sizeof(uint16_t);
}

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

// Ranks the NT*8 items of the CTA: thread (warp w, lane l) passes the value bits v[e] of position
// p = 256 w + 32 e + l and whether that position holds an entry (valid[e]; invalid ones are fills).
// On return (after a barrier) s_item[j] holds the item of rank j, whose low kSlotBits bits are its
// position: valid items by value descending, equal values by position, then the fills by
// position.  `smem` holds rank_smem_bytes<BF16>(NT) bytes, 16-byte aligned; every thread of the
// CTA calls.  The first write to `smem` follows a barrier inside the call, so it may hold data
// that the caller's threads read up to the call.
template <bool BF16, int NT>
__device__ void value_rank(const uint32_t (&v)[kEpt], const bool (&valid)[kEpt], unsigned char *smem)
{
    using K = Item<BF16>;
    constexpr int nt = NT, n_items = NT * kEpt, nw = NT / 32;
    static_assert(n_items <= (1 << kSlotBits), "positions must fit the slot bits");
    __shared__ uint32_t s_red[64];
    K *s_item = reinterpret_cast<K *>(smem);
    uint16_t *s_cnt = reinterpret_cast<uint16_t *>(s_item + n_items);  // [nw][kDigits]
    uint16_t *s_base = s_cnt + nw * kDigits;                              // [kDigits]
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int wbase = warp * kWarpItems;

    uint32_t kp[kEpt], kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
    for (int e = 0; e < kEpt; ++e) {
        kp[e] = BF16 ? inv_key_bf16(v[e]) : inv_key_f32(v[e]);
        if (valid[e]) {
            kmin = min(kmin, kp[e]);
            kmax = max(kmax, kp[e]);
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
        const uint64_t kk = valid[e] ? static_cast<uint64_t>(kp[e] - kmin) : fill_key;
        item[e] = (static_cast<K>(kk) << kSlotBits) | static_cast<K>(wbase + e * 32 + lane);
    }
    const uint32_t lt = lanemask_lt();
    uint16_t *wcnt = s_cnt + warp * kDigits;
    constexpr int dpt = kDigits >= nt ? kDigits / nt : 1;  // digits a thread scans
    __syncthreads();  // every thread has read s_red

    for (int shift = kSlotBits; shift < kSlotBits + bits; shift += kRadixBits) {
        const int nb = min(kRadixBits, kSlotBits + bits - shift);  // digit bits that can be nonzero
        // this warp's counters (the previous pass read them before its closing barrier)
#pragma unroll
        for (int i = lane; i < kDigits; i += 32) wcnt[i] = 0;
        // the lanes holding the same digit in each of the warp's 8 item rows.  Two ways: one
        // ballot per digit bit (a fixed cost), or match, whose cost grows with the number of
        // distinct digits among the lanes.  On wide digits the warp matches its first row and keeps
        // matching when that row held at most kMatchMaxDistinct digits (tie-heavy rows); otherwise,
        // and on narrow digits, ballots.
        uint32_t dg[kEpt], peers[kEpt];
#pragma unroll
        for (int e = 0; e < kEpt; ++e) {
            dg[e] = static_cast<uint32_t>(item[e] >> shift) & (kDigits - 1);
            peers[e] = 0xffffffffu;
        }
        bool matched = false;  // warp-uniform
        if (nb > kBallotOnlyBits) {
            peers[0] = __match_any_sync(0xffffffffu, dg[0]);
            const uint32_t leads = __ballot_sync(0xffffffffu, (peers[0] & lt) == 0u);  // one lane per digit
            matched = __popc(leads) <= kMatchMaxDistinct;
        }
        if (matched) {
#pragma unroll
            for (int e = 1; e < kEpt; ++e) peers[e] = __match_any_sync(0xffffffffu, dg[e]);
        } else {
            const int e0 = nb > kBallotOnlyBits ? 1 : 0;  // row 0 was matched already
#pragma unroll
            for (int b = 0; b < kRadixBits; ++b) {
                if (b < nb) {
#pragma unroll
                    for (int e = 0; e < kEpt; ++e) {
                        if (e < e0) continue;
                        const uint32_t one = (dg[e] >> b) & 1u;
                        // lanes whose bit b equals this lane's: the ballot, inverted when the bit is 0
                        peers[e] &= __ballot_sync(0xffffffffu, one != 0u) ^ (one - 1u);
                    }
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
                wcnt[dg[e]] = static_cast<uint16_t>(base + __popc(peers[e]));
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
                    s_cnt[w * kDigits + d] = static_cast<uint16_t>(run);
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
            if (d < kDigits) s_base[d] = static_cast<uint16_t>(run);
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
}

// Position (0 .. NT*8-1) of the item of rank j after value_rank.
template <bool BF16>
__device__ __forceinline__ int ranked_position(const unsigned char *smem, int j)
{
    return static_cast<int>(reinterpret_cast<const Item<BF16> *>(smem)[j] & ((Item<BF16>(1) << kSlotBits) - 1));
}

}  // namespace order
}  // namespace sel
