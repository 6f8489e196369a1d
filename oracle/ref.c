/*
 * oracle/ref.c -- plain, slow CPU definition of batched row-wise top-k and of
 * the flat row gather.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA path is held
 * to.  Only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg may load it; the product path never calls it and shares no
 * code, header, table or constant generator with it.
 *
 * Sources (web pages; the section each rule comes from):
 *   [DS]  "Speed up PyTorch TopK with DeepSelect" (tutorial):
 *         "Supported workloads"          k <= 4096, bf16 indexer rows, fp32 sampling rows
 *         "Key features"                 int32/int64 indices, optional values,
 *                                        per-row exclusive end, NaN check
 *         "Basic TopK usage"             values have x's dtype; sorted_index =>
 *                                        each row's indices ascending
 *         "Working with variable-length rows"
 *                                        row r uses columns [0, end[r]); a row
 *                                        shorter than k is filled with the
 *                                        out-of-bounds fill values
 *         "NaN handling"                 rows whose valid length is <= k are
 *                                        not checked for NaN
 *   [HP]  MindSpore hyper-parallel pull request "perf/gather-index-select",
 *         description: key[batch, position] equals one index_select over the
 *         batch-flattened key at batch * comp_len + position; positions are
 *         the "safe" (clamped) positions.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): top-k keeps the LARGEST values; among equal values the smaller
 * column index wins; -0 and +0 compare equal (plain float comparison);
 * the index fill is -1 and the value fill is -inf; valid entries come first
 * and fills last; a row holding a NaN (only rows with n > k are checked) is
 * flagged and its selection is left unspecified (the oracle writes fills);
 * a negative gather position reads position 0; a position >= comp_len yields
 * a zero row and is counted as an error.
 *
 * Every comparison is done in double precision on the exact value of the
 * element (fp32 and bf16 convert to double without rounding).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

typedef struct {
    double v;
    int64_t i;
} oracle_item;

static double element_value(const void *x, int dtype, int64_t off, uint32_t *bits_out)
{
    if (dtype == ORACLE_F32) {
        uint32_t u;
        float f;
        memcpy(&u, (const char *)x + 4 * off, 4);
        memcpy(&f, &u, 4);
        *bits_out = u;
        return (double)f;
    } else {
        uint16_t h;
        uint32_t u;
        float f;
        memcpy(&h, (const char *)x + 2 * off, 2);
        u = (uint32_t)h << 16; /* a bf16 number is the upper half of an fp32 */
        memcpy(&f, &u, 4);
        *bits_out = h;
        return (double)f;
    }
}

/* Larger value first; equal values: smaller index first.  A total order on
 * NaN-free rows, so the result does not depend on qsort's stability. */
static int by_value_desc_then_index(const void *a, const void *b)
{
    const oracle_item *p = (const oracle_item *)a;
    const oracle_item *q = (const oracle_item *)b;
    if (p->v > q->v) return -1;
    if (p->v < q->v) return 1;
    if (p->i < q->i) return -1;
    if (p->i > q->i) return 1;
    return 0;
}

/* Value order of the output ("Performance and advanced tips", item 3: results
 * ordered by value): larger value first, equal values by smaller index, and a
 * NaN (only short rows, which are not checked, can keep one) above every
 * number, NaNs among themselves by index. */
static int by_value_nan_first_then_index(const void *a, const void *b)
{
    const oracle_item *p = (const oracle_item *)a;
    const oracle_item *q = (const oracle_item *)b;
    const int pn = p->v != p->v, qn = q->v != q->v;
    if (pn != qn) return pn ? -1 : 1;
    if (!pn) {
        if (p->v > q->v) return -1;
        if (p->v < q->v) return 1;
    }
    return p->i < q->i ? -1 : (p->i > q->i);
}

static int by_index(const void *a, const void *b)
{
    const oracle_item *p = (const oracle_item *)a;
    const oracle_item *q = (const oracle_item *)b;
    return (p->i > q->i) - (p->i < q->i);
}

uint32_t oracle_value_fill_bits(int dtype)
{
    return dtype == ORACLE_F32 ? 0xFF800000u : 0xFF80u; /* -inf */
}

/*
 * Row-wise top-k, written as its definition: sort the valid prefix of each
 * row by (value descending, index ascending) and keep the first k.
 *
 *   x        bit patterns, row-major [rows, stride]; columns [0, cols) hold data
 *   row_end  int32 [rows] exclusive end per row, or NULL (= cols); clamped to [0, cols]
 *   out_idx  int64 [rows, k]       selected column indices, -1 fills
 *   out_bits uint32 [rows, k]      raw bits of the selected values (fp32 bits or
 *                                  the 16 bf16 bits), fills = -inf bits
 *   row_nan  int32 [rows]          1 if the row was checked and holds a NaN
 *
 * sorted_index picks the order of a row's k entries:
 *   0  long rows by value descending (ties by index), short rows by index;
 *   1  by index ascending ("Basic TopK usage");
 *   2  by value descending for every row, equal values by index, a NaN above
 *      every number, fills last.
 * Returns 0, or -1 on bad arguments or allocation failure.
 */
int oracle_topk(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride,
                const int32_t *row_end, int64_t k, int sorted_index,
                int64_t *out_idx, uint32_t *out_bits, int32_t *row_nan)
{
    if (!x || !out_idx || !out_bits || !row_nan || rows < 0 || cols < 0 || stride < cols || k < 1)
        return -1;
    if (sorted_index < 0 || sorted_index > 2)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16)
        return -1;
    oracle_item *items = (oracle_item *)malloc(sizeof(oracle_item) * (size_t)(cols > 0 ? cols : 1));
    if (!items)
        return -1;
    const uint32_t fill = oracle_value_fill_bits(dtype);
    for (int64_t r = 0; r < rows; ++r) {
        int64_t n = cols;
        if (row_end) {
            n = row_end[r];
            if (n < 0) n = 0;
            if (n > cols) n = cols;
        }
        int64_t *oi = out_idx + r * k;
        uint32_t *ob = out_bits + r * k;
        row_nan[r] = 0;
        if (n <= k) {
            /* short row: every valid column, in order (value order in mode 2), then fills;
             * no NaN check */
            for (int64_t j = 0; j < n; ++j) {
                uint32_t bits;
                items[j].v = element_value(x, dtype, r * stride + j, &bits);
                items[j].i = j;
            }
            if (sorted_index == 2)
                qsort(items, (size_t)n, sizeof(oracle_item), by_value_nan_first_then_index);
            for (int64_t j = 0; j < k; ++j) {
                if (j < n) {
                    uint32_t bits;
                    (void)element_value(x, dtype, r * stride + items[j].i, &bits);
                    oi[j] = items[j].i;
                    ob[j] = bits;
                } else {
                    oi[j] = -1;
                    ob[j] = fill;
                }
            }
            continue;
        }
        int has_nan = 0;
        for (int64_t j = 0; j < n; ++j) {
            uint32_t bits;
            double v = element_value(x, dtype, r * stride + j, &bits);
            if (v != v)
                has_nan = 1;
            items[j].v = v;
            items[j].i = j;
        }
        if (has_nan) {
            row_nan[r] = 1;
            for (int64_t j = 0; j < k; ++j) {
                oi[j] = -1;
                ob[j] = fill;
            }
            continue;
        }
        qsort(items, (size_t)n, sizeof(oracle_item), by_value_desc_then_index);
        if (sorted_index == 1)
            qsort(items, (size_t)k, sizeof(oracle_item), by_index);
        for (int64_t j = 0; j < k; ++j) {
            uint32_t bits;
            (void)element_value(x, dtype, r * stride + items[j].i, &bits);
            oi[j] = items[j].i;
            ob[j] = bits;
        }
    }
    free(items);
    return 0;
}

/*
 * Flat row gather: out[r, j, :] = key[b_r, p, :] with b_r = r / (rows / b) and
 * p = max(idx[r, j], 0).  A position >= comp_len gives a zero row and is
 * counted.
 *
 *   key      uint16 bit patterns, element (bb, p, e) at
 *            bb * key_batch_stride + p * key_row_stride + e
 *   idx      int64, element (r, j) at r * idx_row_stride + j
 *   out      uint16 [rows, n, d] contiguous
 *
 * Returns the number of out-of-range positions, or -1 on bad arguments.
 */
int64_t oracle_gather_rows(const uint16_t *key, int64_t b, int64_t comp_len, int64_t d,
                           int64_t key_batch_stride, int64_t key_row_stride,
                           const int64_t *idx, int64_t rows, int64_t n, int64_t idx_row_stride,
                           uint16_t *out)
{
    if (!key || !idx || !out || b < 1 || rows < 0 || rows % b != 0 || n < 0 || d < 1)
        return -1;
    const int64_t rows_per_batch = rows / b;
    int64_t bad = 0;
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t bb = r / rows_per_batch;
        for (int64_t j = 0; j < n; ++j) {
            int64_t p = idx[r * idx_row_stride + j];
            uint16_t *o = out + (r * n + j) * d;
            if (p < 0)
                p = 0;
            if (p >= comp_len) {
                ++bad;
                for (int64_t e = 0; e < d; ++e)
                    o[e] = 0;
                continue;
            }
            for (int64_t e = 0; e < d; ++e)
                o[e] = key[bb * key_batch_stride + p * key_row_stride + e];
        }
    }
    return bad;
}
