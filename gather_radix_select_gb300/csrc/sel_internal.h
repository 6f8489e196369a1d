// sel_internal.h -- argument blocks and launcher declarations shared by the
// C-ABI layer (api.cu) and the kernels (topk.cu, gather.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace sel {

// Debug builds (-DSEL_DEBUG: the library libsel_debug.so) check selected accesses before they are
// made -- staged-list and region offsets, workspace slots, output positions, gathered key rows.
// SEL_IN_BOUNDS(cond, flag) is true when the access may go ahead; otherwise the access is skipped
// and kStatusBounds (SEL_EBOUNDS) goes to *flag (the first nonzero status wins).  Normal builds
// compile every check away (cond is not evaluated).
constexpr int32_t kStatusBounds = 7;
#if defined(__CUDACC__) && defined(SEL_DEBUG)
__device__ __forceinline__ bool bounds_ok(bool ok, int32_t *flag)
{
    if (!ok && flag) atomicCAS(flag, 0, kStatusBounds);
    return ok;
}
#define SEL_IN_BOUNDS(cond, flag) (::sel::bounds_ok((cond), (flag)))
#else
#define SEL_IN_BOUNDS(cond, flag) true
#endif

constexpr int kMaxLevels = 4;       // radix passes (digits) at most
constexpr int kMaxSlice = 65536;    // elements of a row staged by one CTA (list offsets are 16-bit)
constexpr int kMaxChunks = 16;      // bulk-copy chunks per CTA slice
constexpr uint32_t kChunkBytes = 16384;
constexpr int kWideStage = 64;              // wide_kernel: staged candidate vectors per warp
constexpr int kWideSampleVecsPerLane = 2;  // wide_kernel: 16-byte vectors per lane in the threshold sample
constexpr int kWideThreads = 512;
constexpr int kMaxParts = 64;       // CTAs splitting one row (split_kernel)
constexpr int kModeRow = 0;         // row_kernel: one CTA per row, row staged in shared memory
constexpr int kModeSplit = 1;       // split_kernel: `parts` CTAs per row + last-arriver merge
constexpr int kModeStream = 2;      // stream_kernel: one CTA per row, passes read global memory
constexpr int kModeWide = 3;        // wide_kernel: one CTA per row, one streaming pass into per-warp lists
constexpr int kModeReg2 = 4;        // reg_kernel: one CTA per row held in registers, 2 vectors a thread
constexpr int kModeReg8 = 5;        // reg_kernel: 8 vectors a thread
constexpr int kModeWideSplit = 6;   // wide_kernel over `parts` CTAs per row, last-arriver merge
constexpr int kModeFlat = 7;        // flat_kernel: rows cut into chunks dealt over a persistent grid
constexpr int kModeRowOrdered = 8;  // row_kernel that also ranks each row's outputs by value
constexpr int kModeReg2Ordered = 9; // reg_kernel (2 vectors a thread) ranking its outputs by value
constexpr int kModeReg8Ordered = 10; // reg_kernel (8 vectors a thread) ranking its outputs by value
constexpr int kNumModes = 11;
// flat_kernel: warps 0..23 stream, warps 24..31 estimate thresholds, flush chunks and select
constexpr int kFlatStreamWarps = 24;
constexpr int kFlatSelWarps = 8;
constexpr int kFlatThreads = (kFlatStreamWarps + kFlatSelWarps) * 32;
constexpr int kFlatQueue = 64;        // chunks of one CTA at most
constexpr int kFlatMaxParts = 64;     // chunks of one row at most
constexpr int kFlatBufs = 3;          // chunk buffers in shared memory, in rotation
constexpr int kFlatSampleVecs = 1024; // row sample for the threshold estimate: 32 runs of 32 vectors
constexpr int kGatherThreads = 256;

// Everything one selection launch needs; passed by value (kernel parameter space).
struct TopkArgs {
    const void *x;            // [rows, stride] elements (fp32 or bf16 bits)
    int64_t rows, cols, stride;
    const int32_t *row_end;   // nullable
    int64_t row_end_div;      // > 1: a row has ceil(row_end / row_end_div) valid columns
    int32_t row_order;        // 1: CTA (or CTA group) b takes row b/2 (b even) or rows - 1 - b/2 (b odd)
    int32_t k;
    int32_t idx_i64;          // 0: int32 indices, 1: int64
    int32_t want_values;
    void *out_idx;            // nullable only in the fused launch
    int64_t out_idx_stride;
    void *out_val;            // nullable
    int64_t out_val_stride;
    int32_t *nan_flag;        // nullable
    int32_t *err_flag;        // nullable
    int64_t slice;            // elements of a row per CTA (multiple of 64); flat_kernel: 16-byte vectors per chunk
    int32_t parts;            // CTAs per row (split_kernel); chunks per row (flat_kernel)
    int32_t nlevels;          // digits from the most significant end
    int32_t bits[kMaxLevels];
    int32_t hist_bins;        // 1 << max(bits)
    uint32_t smem_buf_bytes;  // bytes reserved for the staged slice
    uint32_t smem_hist_off;   // offset of the local histogram
    uint32_t smem_mask_off;   // offset of the per-vector candidate masks (one byte per 16-byte vector)
    uint32_t smem_list_off;   // offset of the candidate list (16-bit offsets within the slice)
    uint32_t smem_glist_off;  // offset of the gather position list (fused only)
    uint32_t smem_stage_off;  // wide_kernel, flat_kernel: staged candidate vectors
    uint32_t smem_order_off;  // row / reg kernel ranked by value: the ranking's items and counters
    uint32_t smem_cbuf_off;   // flat_kernel: chunk buffers
    int32_t flat_wcap;        // flat_kernel: pairs one streaming warp may keep of one chunk
    int32_t flat_sel_pairs;   // flat_kernel: pairs the selection regions hold in all
    int32_t list_cap;         // capacity of the candidate list
    int32_t region_stride;    // wide_kernel: candidate pairs per warp region (capacity list_cap + 1)
    int32_t part_cap;         // wide_kernel over parts: candidate pairs a part may leave in the workspace;
                              // flat_kernel: pairs one streaming warp may leave for one chunk
    int32_t agg;              // 1: first-pass histogram with warp-aggregated atomics
    int32_t sample_step;      // > 1: the first digit's threshold is estimated from every
                              //      sample_step-th 16-byte vector of the row
    int32_t sample_min_cols;  // rows shorter than this use the exact first histogram
    // split_kernel workspace (see topk_impl.cuh for the layout)
    unsigned char *ws;
    size_t ws_bytes;          // the workspace's size (debug-build checks)
    int64_t ws_counter_bytes, ws_row_bytes, ws_head_bytes, ws_part_bytes, ws_bits_bytes;
    // fused gather (ignored unless the gather variant is launched)
    const uint16_t *key;
    int64_t comp_len, d, key_batch_stride, key_row_stride, rows_per_batch;
    int64_t key_span;         // elements from key[0] to the end of its last row (debug-build checks)
    int64_t n_gather;
    uint16_t *gather_out;     // [rows, n_gather, d]
};

struct GatherArgs {
    const uint16_t *key;
    int64_t comp_len, d, key_batch_stride, key_row_stride;
    int64_t key_span, key2_span;  // elements from key[0] (key2[0]) to the end of its last row (debug checks)
    const void *idx;
    int32_t idx_i64;
    int64_t rows, n, idx_row_stride, rows_per_batch;
    uint16_t *out;
    // optional second key gathered at the same positions (same b and comp_len); out2 null = none
    const uint16_t *key2;
    int64_t d2, key2_batch_stride, key2_row_stride;
    uint16_t *out2;
    int32_t *err_flag;
    int64_t pairs_per_cta;    // (row, position) pairs handled by one CTA
    int32_t ctas_per_row;
};

// Expansion of selected blocks to positions, with the gather of their key rows (gather.cu).
constexpr int kBlockSelectMax = 128;  // block_expand_kernel selects rows of at most this many blocks itself

struct BlockArgs {
    int32_t *pos;             // [rows, pos_stride]: selected block ids in [0, topk_blocks) on entry
    int64_t pos_stride;       //   (unless scores is set), their valid positions ascending then -1 on exit
    // set: the kernel selects the blocks itself from these scores (n_blocks <= kBlockSelectMax)
    const void *scores;
    int32_t scores_bf16;
    int64_t n_blocks, scores_stride;
    int32_t *nan_flag;
    int64_t rows;
    int32_t topk_blocks;
    int64_t block_size;
    const int32_t *pos_end;   // nullable: exclusive end of each row's valid positions
    int64_t pos_limit;        // n_blocks * block_size (the end when pos_end is null)
    // gather (key null = none), as GatherArgs
    const uint16_t *key;
    int64_t comp_len, d, key_batch_stride, key_row_stride, rows_per_batch;
    int64_t key_span;
    uint16_t *out;            // [rows, topk_blocks * block_size, d]
    int32_t *err_flag;
    int32_t ctas_per_row;     // set by the launcher: several only when the kernel selects the blocks
};

cudaError_t launch_block_expand(const BlockArgs &a, cudaStream_t stream);

// Re-ordering of finished output rows by value (order.cu).
struct OrderArgs {
    const void *x;            // the selection's input rows (values are read here when out_val is null)
    int64_t x_stride;         // elements
    int64_t rows;
    int32_t k;
    void *out_idx;            // [rows, out_idx_stride] int32 or int64
    int64_t out_idx_stride;
    void *out_val;            // nullable: [rows, out_val_stride] value bits
    int64_t out_val_stride;
    // optional gather of the first n_gather ordered positions (n_gather 0: none), as gather_kernel:
    // gather_out[r, j, :] = key[r / rows_per_batch, max(idx[r, j], 0), :]
    const uint16_t *key;
    int64_t comp_len, d, key_batch_stride, key_row_stride, rows_per_batch, key_span;
    int64_t n_gather;
    uint16_t *gather_out;     // [rows, n_gather, d]
    int32_t *err_flag;        // nullable: SEL_EINVAL for a position past comp_len (zero row written)
};

// dtype: 0 fp32, 1 bf16.  Sorts each output row by value descending (ties: column ascending), then
// gathers the first n_gather ordered positions' key rows when n_gather > 0.
cudaError_t launch_value_order(int dtype, bool idx_i64, const OrderArgs &a, cudaStream_t stream);

// dtype: 0 fp32, 1 bf16.  mode: one of the kMode* values.  grid: CTAs to launch.
cudaError_t launch_topk(int dtype, int mode, int threads, bool gather, size_t smem_bytes, const TopkArgs &a,
                        int64_t grid, cudaStream_t stream);

// CTAs of that kernel configuration that fit on one SM (0 = cannot launch).
int topk_blocks_per_sm(int dtype, int mode, int threads, bool gather, size_t smem_bytes);

// Per element type (topk_f32.cu / topk_bf16.cu).
cudaError_t launch_topk_f32(int mode, int threads, bool gather, size_t smem, const TopkArgs &a, cudaStream_t s,
                            int64_t grid, bool query, int *blocks_per_sm);
cudaError_t launch_topk_bf16(int mode, int threads, bool gather, size_t smem, const TopkArgs &a, cudaStream_t s,
                             int64_t grid, bool query, int *blocks_per_sm);

// One CTA whose bounded mbarrier wait runs out after `cycles` (test of the timeout path).
cudaError_t launch_wait_selftest(int32_t *err_flag, long long cycles, cudaStream_t s);

// Max dynamic shared memory a selection CTA may use on the current device.
size_t topk_smem_limit();

cudaError_t launch_gather(const GatherArgs &a, cudaStream_t stream);

int device_sm_count();

// sel_topk's host-side argument checks (api.cu), for entry points that wrap it.
int check_topk_call(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride, int k, int sorted_index,
                    int idx_dtype, int want_values, const void *out_idx, int64_t out_idx_stride, const void *out_val,
                    int64_t out_val_stride);

}  // namespace sel
