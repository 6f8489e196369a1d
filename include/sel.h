/*
 * sel.h -- C ABI of libsel: batched row-wise top-k selection and the flat
 * row gather of the selected key rows, on one GB300 (sm_103a).
 *
 * Operations and the passages that define them:
 *
 *   sel_topk          "Speed up PyTorch TopK with DeepSelect" (tutorial):
 *                     "Basic TopK usage" (2-D input, contiguous last dim,
 *                     values in x's dtype, int32/int64 indices, sorted_index
 *                     = ascending indices per row), "Returning indices only"
 *                     (return_value=False), "Working with variable-length
 *                     rows" (per-row exclusive end, fills for rows shorter
 *                     than k), "NaN handling" (rows with valid length <= k are
 *                     not checked), "Supported workloads" (k <= 4096).
 *   sel_stride_requirement
 *                     same tutorial, "Handling stride alignment" (input and
 *                     output row-stride alignment in bytes).
 *   sel_gather_rows   MindSpore hyper-parallel pull request
 *                     "perf/gather-index-select", description: the gather
 *                     key[batch, position] done as one index_select over the
 *                     batch-flattened key at batch * comp_len + position,
 *                     with clamped ("safe") positions.
 *   sel_topk_gather   the two above in one launch: the selection's index list
 *                     feeds the gather without a round trip through memory.
 *   sel_gather_rows_pair
 *                     the same pull request: the Indexer KL loss gathers the
 *                     index key and the attention key at one index list;
 *                     both gathers in one launch.
 *   sel_block_topk_gather
 *                     the same pull request: the compressed_candidate_topk
 *                     chain -- top blocks of compressed positions, expanded
 *                     to topk_blocks * block_size positions, sorted, masked
 *                     and gathered.
 *   sel_topk_noalloc  sel_topk with its scratch in a built-in device array.
 *   sel_topk_workspace_size, sel_max_cols, sel_topk_kernel_name, sel_strerror
 *                     queries (no device work).
 *
 * Value order (sorted_index = SEL_SORT_VALUE; the tutorial's "Performance
 * and advanced tips", item 3, names ordering by index or by value) is ranked
 * inside the selection launch where the selection kernel holds the row's
 * selected columns in shared memory (the staged row kernel; the register
 * kernel when the call also gathers), else in one extra launch.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     allocates no device memory on any call (it keeps small host-side caches
 *     of launch plans).  Scratch, where a shape needs it, is a caller-owned
 *     workspace (sel_topk_workspace_size), or the built-in array of
 *     sel_topk_noalloc.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  No call synchronises.
 *   - The return value is a sel_status.  Argument errors are found on the
 *     host before anything is launched.  Findings made on the device are
 *     written to caller-owned int32 flags: `nan_flag` is OR-ed with 1 when a
 *     checked row holds a NaN; `err_flag` receives a nonzero sel_status
 *     (first writer wins) when a device wait timed out or a gather position
 *     was out of range.  Both flags are optional (NULL) and must be zeroed by
 *     the caller.  Nothing traps.
 *   - Element strides are in ELEMENTS, not bytes.
 *   - Reads stay inside [0, row_end) of each input row; padding columns and
 *     pad rows are never read.
 *
 * Readings of the tutorial where it is silent (stated once here):
 *   - "top-k" keeps the LARGEST values; among equal values the smaller
 *     column index wins; -0.0 and +0.0 are equal.
 *   - Index fill is -1; value fill is -inf (fp32 0xFF800000, bf16 0xFF80).
 *     Valid entries come first, fills last.
 *   - Without sorted_index the order of a row's k entries is unspecified
 *     (this implementation happens to return them in ascending index order).
 *   - A NaN is not trapped: it sets *nan_flag and the selection of that row
 *     is unspecified (but only in-range indices are written).
 */
#ifndef SEL_H_
#define SEL_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SEL_API __attribute__((visibility("default")))
#else
#define SEL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SEL_OK = 0,
    SEL_EINVAL = 1,       /* bad argument (k, sizes, null pointer, gather position) */
    SEL_EALIGN = 2,       /* a pointer or row stride breaks the alignment rule */
    SEL_EUNSUPPORTED = 3, /* dtype / width outside what the kernels handle */
    SEL_ECUDA = 4,        /* a CUDA runtime call failed (launch, attribute query) */
    SEL_ETIMEOUT = 5,     /* (device flag only) a bounded device wait ran out */
    SEL_ESCRATCH = 6,     /* sel_topk_noalloc: the shape needs more scratch than the built-in array */
    SEL_EBOUNDS = 7       /* (device flag, debug build only) an out-of-bounds access was caught and skipped */
} sel_status;

enum { SEL_F32 = 0, SEL_BF16 = 1 };  /* input element type */
enum { SEL_I32 = 0, SEL_I64 = 1 };   /* index element type */
/* Order of a row's k entries (the sorted_index argument; "Performance and
 * advanced tips", item 3: results ordered by index or by value). */
enum { SEL_UNSORTED = 0, SEL_SORT_INDEX = 1, SEL_SORT_VALUE = 2 };

#define SEL_MAX_K 4096

/* Alignment contract ("Handling stride alignment").  *in_align_bytes: the
 * input base pointer and the input row stride in bytes must be multiples of
 * it (rows are staged into shared memory by bulk copies).  *out_align_bytes:
 * every output base pointer and output row stride in bytes must be multiples
 * of it, so outputs of small k come with padded (non-contiguous) rows.
 * Either pointer may be NULL.  Always returns SEL_OK. */
SEL_API int sel_stride_requirement(int *in_align_bytes, int *out_align_bytes);

/* Row-wise top-k.
 *   x           [rows, stride] elements of `dtype` (SEL_F32 | SEL_BF16); the first
 *               `cols` of each row are data.  Needs stride >= cols.
 *   row_end     int32 [rows] exclusive end per row, clamped on the device to
 *               [0, cols]; NULL means cols for every row.
 *   k           1..SEL_MAX_K.  k > cols is allowed (every row is then short).
 *   sorted_index  SEL_UNSORTED: any order.  SEL_SORT_INDEX: each row's indices
 *               ascending (values follow).  SEL_SORT_VALUE: values descending,
 *               equal values by index ascending, fills last; a NaN (possible
 *               only in a short row, which is not checked) counts above every
 *               number.  Value order takes one launch where the plan is the
 *               staged row kernel, else a second launch after the selection.
 *   idx_dtype   SEL_I32 | SEL_I64.
 *   out_idx     [rows, out_idx_stride] of idx_dtype; columns [0, k) written.
 *   out_val     [rows, out_val_stride] of `dtype`, or NULL when want_values == 0.
 *   workspace   device scratch of at least sel_topk_workspace_size(dtype, rows,
 *               cols, k) bytes, 256-byte aligned, any contents (its counters
 *               are cleared on `stream` by the call); may be NULL when that
 *               size is 0.  Calls that run at the same time need separate
 *               workspaces.
 *   nan_flag, err_flag   optional device int32 flags (see above).
 * Errors: SEL_EINVAL (k out of range, negative sizes, stride < cols, output
 * strides < k, null required pointer, bad enum, missing or short workspace),
 * SEL_EALIGN, SEL_EUNSUPPORTED (cols > 2^31 - 1), SEL_ECUDA (launch failure).
 * rows == 0 returns SEL_OK without a launch. */
SEL_API int sel_topk(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride,
             const int32_t *row_end, int k, int sorted_index, int idx_dtype, int want_values,
             void *out_idx, int64_t out_idx_stride, void *out_val, int64_t out_val_stride,
             void *workspace, size_t workspace_bytes,
             int32_t *nan_flag, int32_t *err_flag, void *stream);

/* Scratch bytes sel_topk / sel_topk_gather need for this shape on the current
 * device: non-zero only when few rows are wide enough to be split over several
 * CTAs, whose candidate lists meet in the workspace.  0 on invalid arguments. */
SEL_API size_t sel_topk_workspace_size(int dtype, int64_t rows, int64_t cols, int k);

/* Largest `cols` sel_topk accepts for `dtype` (indices must fit int32). */
SEL_API int64_t sel_max_cols(int dtype);

/* Name of the kernel a sel_topk (n_gather == 0) or sel_topk_gather call of this
 * shape launches on the current device: "reg_kernel", "row_kernel",
 * "wide_kernel", "split_kernel" or "stream_kernel" (static strings, never freed), or NULL on
 * invalid arguments.  A diagnostic for profiling and reports; it launches
 * nothing.  The tutorial has no counterpart: it is this library's own plan. */
SEL_API const char *sel_topk_kernel_name(int dtype, int64_t rows, int64_t cols, int k, int64_t n_gather);

/* Flat row gather:  out[r, j, :] = key[b_r, max(idx[r, j], 0), :],
 * b_r = r / (rows / b).
 *   key         bf16 element (bb, p, e) at bb*key_batch_stride + p*key_row_stride + e;
 *               rows of the key may be strided (non-contiguous key).
 *   idx         idx_dtype element (r, j) at r*idx_row_stride + j.
 *   rows        a multiple of b (rows are batch-major).
 *   out         bf16 [rows, n, d] contiguous.
 * A negative position reads position 0; a position >= comp_len writes a zero
 * row and sets *err_flag = SEL_EINVAL.  Alignment: key, out and the key
 * strides must make every key row and out row start on 16 bytes, and
 * d*2 must be a multiple of 16 (else SEL_EALIGN). */
SEL_API int sel_gather_rows(const void *key, int64_t b, int64_t comp_len, int64_t d,
                    int64_t key_batch_stride, int64_t key_row_stride,
                    const void *idx, int idx_dtype, int64_t rows, int64_t n, int64_t idx_row_stride,
                    void *out, int32_t *err_flag, void *stream);

/* Two flat row gathers at the same positions, in one launch (MindSpore
 * hyper-parallel pull request "perf/gather-index-select": the Indexer KL loss
 * gathers the index key and the attention key with one index list):
 *     out [r, j, :] = key [b_r, max(idx[r, j], 0), :]   (d  elements a row)
 *     out2[r, j, :] = key2[b_r, max(idx[r, j], 0), :]   (d2 elements a row)
 * Both keys are bf16 [b, comp_len, *] with their own strides; every argument
 * means what it means in sel_gather_rows, and the same checks apply to each
 * key.  A position >= comp_len gives zero rows in both outputs and sets
 * err_flag = SEL_EINVAL. */
SEL_API int sel_gather_rows_pair(const void *key, int64_t d, int64_t key_batch_stride, int64_t key_row_stride,
                                 const void *key2, int64_t d2, int64_t key2_batch_stride, int64_t key2_row_stride,
                                 int64_t b, int64_t comp_len, const void *idx, int idx_dtype, int64_t rows, int64_t n,
                                 int64_t idx_row_stride, void *out, void *out2, int32_t *err_flag, void *stream);

/* Block-level candidate selection with its gather (MindSpore hyper-parallel
 * pull request "perf/gather-index-select": the `compressed_candidate_topk`
 * chain picks the top blocks of compressed positions, expands them to
 * topk_blocks * block_size positions, sorts and masks the positions, and
 * gathers the key rows there -- its Index, Sort and MaskedFill steps):
 *   scores      [rows, stride] block scores of `dtype`, n_blocks columns; block
 *               c covers positions [c * block_size, (c + 1) * block_size).
 *   pos_end     int32 [rows]: exclusive end of each row's valid positions,
 *               clamped on the device to [0, n_blocks * block_size]; NULL
 *               means n_blocks * block_size.  A block is a candidate when it
 *               holds a valid position.
 *   topk_blocks 1..SEL_MAX_K blocks chosen per row by sel_topk's rule (largest
 *               score, smaller block first on ties; fewer candidates than
 *               topk_blocks: all of them).
 *   out_pos     int32 [rows, out_pos_stride], out_pos_stride >= topk_blocks *
 *               block_size (alignment as sel_topk's out_idx): the chosen
 *               blocks' valid positions, ascending, then -1.
 *   key .. key_row_stride, gather_out   as sel_gather_rows, gathering
 *               out_pos (a -1 reads position 0); key and gather_out both
 *               NULL: positions only.
 *   workspace, nan_flag, err_flag       as sel_topk (shape rows x n_blocks,
 *               k = topk_blocks).
 * One launch for rows of at most 128 blocks (the expansion kernel ranks the
 * blocks itself); wider rows take two (sel_topk's selection, then the
 * expansion with the gather). */
SEL_API int sel_block_topk_gather(const void *scores, int dtype, int64_t rows, int64_t n_blocks, int64_t stride,
                                  const int32_t *pos_end, int topk_blocks, int64_t block_size, int32_t *out_pos,
                                  int64_t out_pos_stride, const void *key, int64_t b, int64_t comp_len, int64_t d,
                                  int64_t key_batch_stride, int64_t key_row_stride, void *gather_out,
                                  void *workspace, size_t workspace_bytes, int32_t *nan_flag, int32_t *err_flag,
                                  void *stream);

/* sel_topk followed by sel_gather_rows of the first n_gather output columns
 * (n_gather <= k), in one launch.  The top-k arguments are those of
 * sel_topk (out_idx may be NULL when the indices themselves are not needed);
 * the gather arguments are those of sel_gather_rows with idx taken from the
 * selection.  Fill positions (-1) of short rows gather position 0, as in
 * sel_gather_rows.  The workspace rule is that of sel_topk.  With
 * SEL_SORT_VALUE the gathered columns are those of the value-ordered output
 * (the n_gather largest values); that takes one launch where the plan is
 * the staged row or register kernel, else two (the selection, then one
 * launch that orders each row and gathers its first n_gather ordered
 * positions), and out_idx must not be NULL. */
SEL_API int sel_topk_gather(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride,
                    const int32_t *row_end, int k, int sorted_index, int idx_dtype, int want_values,
                    void *out_idx, int64_t out_idx_stride, void *out_val, int64_t out_val_stride,
                    const void *key, int64_t b, int64_t comp_len, int64_t d,
                    int64_t key_batch_stride, int64_t key_row_stride, int64_t n_gather,
                    void *gather_out, void *workspace, size_t workspace_bytes,
                    int32_t *nan_flag, int32_t *err_flag, void *stream);

/* Size of the device array sel_topk_noalloc takes its scratch from (32 MiB). */
#define SEL_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* sel_topk without a workspace argument, for callers that cannot allocate
 * device memory (for example code running while a framework has reserved the
 * whole device pool for itself, or a C caller with no device allocator).
 * There is no counterpart on the pages this library follows: it is an
 * addition of this library.
 *   Arguments, results and errors are those of sel_topk.  Shapes for which
 *   sel_topk_workspace_size exceeds SEL_NOALLOC_SCRATCH_BYTES are rejected
 *   with SEL_ESCRATCH before anything is launched; use sel_topk with a
 *   workspace for those.
 *   Argument errors (SEL_EINVAL, SEL_EALIGN) are reported before SEL_ESCRATCH.
 *   The scratch is one file-scope device array per GPU, loaded with the
 *   library and held until the process exits; nothing is allocated by the
 *   call.  The array's device address is looked up (with the device current)
 *   on every call whose stream is not capturing a graph, so a device reset
 *   or another current context is picked up; a call made while `stream`
 *   captures reuses the address the last non-capturing call on that device
 *   found.  So after a device reset make one ordinary call before capturing.
 *   Every call shares the array and it keeps the previous call's contents:
 *   the counters that must start at zero are cleared on `stream` by each call.
 *   Calls that overlap on the GPU (other streams, other host threads) race on
 *   the array and give undefined results: serialise them. */
SEL_API int sel_topk_noalloc(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride,
                     const int32_t *row_end, int k, int sorted_index, int idx_dtype, int want_values,
                     void *out_idx, int64_t out_idx_stride, void *out_val, int64_t out_val_stride,
                     int32_t *nan_flag, int32_t *err_flag, void *stream);

/* Static message for a sel_status value. */
SEL_API const char *sel_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* SEL_H_ */
