/*
 * Exact per-row top-k of BF16 logits: the plain CPU definition.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the oracle the CUDA path is checked
 * against. Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * load it; the product library never does, and the two share no code.
 *
 * What it computes follows the vLLM page "decode_topk_cute" (module docstring,
 * "What this module computes"):
 *   - for each row, the indices of its k largest elements, in any order; exact:
 *     every index whose value exceeds the k-th largest, then enough of those
 *     equal to it;
 *   - a row of at most k elements returns 0 .. n-1 and -1 padding, without
 *     looking at the values;
 *   - token mode: an element is one BF16 logit;
 *   - block mode: an element is the NaN-propagating maximum of an aligned group
 *     of 8 logits; the row's newest block is pinned at +inf, and blocks that
 *     score -inf are written as -1;
 *   - values are compared through an order-preserving 16-bit key of their BF16
 *     bits, so ties are exact.
 * The key is the one the sglang PR #39305 page ("Exact bf16 consumer top-k
 * adapted from DeepSelect", Modifications) writes as x ^ (x < 0 ? 0xFFFF :
 * 0x8000): negatives reversed and below the positives, -0 below +0.
 * Ties at the threshold go to the lowest indices (vLLM kimi_k3 "dsa/indexer"
 * page, module docstring, IndexerSelect paragraph).
 * NaN elements are never selected (sglang PR #39305, Modifications).
 * The block-table transform is the one of IndexerSelect.emit on the kimi_k3
 * indexer page: physical = table[row][i / page] * page + i % page.
 *
 * Readings where the pages leave a step open:
 *   - valid_len outside [0, width] is clamped to that range;
 *   - when a row has more than k elements but fewer than k non-NaN ones, the
 *     result is every non-NaN element followed by -1 padding;
 *   - the newest block is pinned even when its group holds a NaN;
 *   - the maximum of {-0, +0} is +0 (the larger key).
 *
 * Method: for every candidate, one 64-bit word (key << 32) | (0xFFFFFFFF - i);
 * sorting those words in descending order sorts by key descending, then index
 * ascending. The first min(k, candidates) words are the selection.
 *
 * The ordered variant follows IndexerSelect on the kimi_k3 indexer page (class
 * docstring and write_selected): the same selected set, written in ascending
 * element-index order ("key order": the page's keys are token positions), -1
 * past the row's count, the count itself per row, and optionally the
 * untransformed indices in the same order. Token mode (the page's logits are
 * one score per token). Reading: the ids past the count are -1, like out.
 *
 * The words variant follows IndexerLocalTopk on the same page (class
 * docstring and candidate): the local top-n of a token row as the DCP merge's
 * B' words, out[r][j] = (key << 16) | (0xFFFF - (l & 0xFFFF)) for the j-th
 * selected element l (0: empty), bit j % 32 of out[r][n + j / 32] = bit 16 of
 * l, valid[r] = the count. Order: the selected elements whose key exceeds the
 * n-th largest key, in index order, then the ties at it that are taken (the
 * lowest indices), in index order. A row of at most n elements takes all of
 * them in index order (their words hold their keys, whatever the values).
 * Readings: NaN elements of longer rows are never selected; when fewer than n
 * are eligible, all of them are taken, in index order.
 *
 * The scorer's "tops" (IndexerScore.rows_out on the same page: each aligned
 * group of 8 logits' largest order key) are defined here over the eligible
 * elements of the group: below the row's valid length and not NaN; a group with
 * none has top 0 (no key is 0, which is below every key a BF16 value has other
 * than the NaN patterns: order_key never yields 0 for a non-NaN value since
 * order_key(0xFFFF) = 0 and 0xFFFF is a NaN).
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_TOKEN = 0, ORACLE_BLOCK8 = 1 };

/* Order-preserving 16-bit key (sglang PR #39305, "distorted" value order). */
static uint16_t order_key(uint16_t x) {
    return (uint16_t)(x ^ ((x & 0x8000u) ? 0xFFFFu : 0x8000u));
}

/* BF16 NaN: exponent all ones and a non-zero mantissa. */
static int is_nan_bf16(uint16_t x) { return (x & 0x7FFFu) > 0x7F80u; }

static const uint16_t KEY_POS_INF = 0xFF80u; /* order_key(0x7F80), +inf */
static const uint16_t KEY_NEG_INF = 0x007Fu; /* order_key(0xFF80), -inf */

static int cmp_desc_u64(const void *a, const void *b) {
    uint64_t x = *(const uint64_t *)a, y = *(const uint64_t *)b;
    return x < y ? 1 : (x > y ? -1 : 0);
}

typedef struct {
    const uint16_t *logits;
    int64_t row_stride;
    int32_t rows, width;
    const int32_t *valid_len;
    int32_t k, mode;
    const int32_t *table;
    int32_t table_stride, page;
    int32_t block_rows, rows_per_request;
    int32_t *out;
    int32_t first_row, row_step;
    int status;
    int ordered;     /* 1: ascending index order, counts in valid, indices in ids */
    int32_t *valid;  /* [rows] when ordered */
    int32_t *ids;    /* [rows, k] or NULL, when ordered */
} job_t;

/* The element index of a candidate word (key << 32) | (0xFFFFFFFF - i). */
static int32_t cand_index(uint64_t w) { return (int32_t)(0xFFFFFFFFu - (uint32_t)w); }

static int cmp_asc_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return x < y ? -1 : (x > y ? 1 : 0);
}

/* Ordered output of the selected logical indices sel_idx[0 .. sel) (sorted in
   place): out and ids in ascending index order, -1 past the count. */
static void write_ordered(const job_t *j, int32_t r, int32_t *sel_idx, int32_t sel);

/* Block-table transform of a logical element index (vLLM kimi_k3 "dsa/indexer",
 * IndexerSelect: a row belongs to request row / q, whose table row it reads;
 * IndexerSelect.emit: the page's id times the physical rows per page, plus the
 * element's offset in its page). */
static int32_t transform(const job_t *j, int32_t r, int32_t i) {
    if (!j->table) return i;
    const int32_t request = r / j->rows_per_request;
    const int64_t page_id = j->table[(int64_t)request * j->table_stride + i / j->page];
    return (int32_t)(page_id * j->block_rows + i % j->page);
}

static int one_row(const job_t *j, int32_t r) {
    const uint16_t *row = j->logits + (int64_t)r * j->row_stride;
    int32_t *out = j->out + (int64_t)r * j->k;
    int32_t L = j->valid_len[r];
    if (L < 0) L = 0;
    if (L > j->width) L = j->width;
    int32_t n = (j->mode == ORACLE_BLOCK8) ? (L + 7) / 8 : L;

    if (n <= j->k) { /* short row: 0 .. n-1 then -1, values never read */
        for (int32_t s = 0; s < j->k; ++s) out[s] = s < n ? transform(j, r, s) : -1;
        if (j->ordered) {
            j->valid[r] = n;
            if (j->ids)
                for (int32_t s = 0; s < j->k; ++s) j->ids[(int64_t)r * j->k + s] = s < n ? s : -1;
        }
        return 0;
    }

    uint64_t *cand = (uint64_t *)malloc((size_t)n * sizeof(uint64_t));
    if (!cand) return 1;
    int32_t m = 0;
    for (int32_t i = 0; i < n; ++i) {
        uint16_t key;
        if (j->mode == ORACLE_TOKEN) {
            uint16_t x = row[i];
            if (is_nan_bf16(x)) continue;
            key = order_key(x);
        } else {
            int nan = 0;
            key = 0;
            int32_t end = 8 * i + 8 < L ? 8 * i + 8 : L;
            for (int32_t t = 8 * i; t < end; ++t) {
                if (is_nan_bf16(row[t])) nan = 1;
                else if (order_key(row[t]) > key) key = order_key(row[t]);
            }
            if (i == n - 1) { nan = 0; key = KEY_POS_INF; } /* newest block */
            if (nan) continue;
        }
        cand[m++] = ((uint64_t)key << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)i);
    }
    qsort(cand, (size_t)m, sizeof(uint64_t), cmp_desc_u64);

    int32_t sel = m < j->k ? m : j->k;
    if (j->ordered) {
        int32_t *sel_idx = (int32_t *)malloc((size_t)(sel > 0 ? sel : 1) * sizeof(int32_t));
        if (!sel_idx) { free(cand); return 1; }
        for (int32_t s = 0; s < sel; ++s) sel_idx[s] = cand_index(cand[s]);
        write_ordered(j, r, sel_idx, sel);
        free(sel_idx);
        free(cand);
        return 0;
    }
    for (int32_t s = 0; s < sel; ++s) {
        uint16_t key = (uint16_t)(cand[s] >> 32);
        int32_t i = cand_index(cand[s]);
        if (j->mode == ORACLE_BLOCK8 && key == KEY_NEG_INF) out[s] = -1;
        else out[s] = transform(j, r, i);
    }
    for (int32_t s = sel; s < j->k; ++s) out[s] = -1;
    free(cand);
    return 0;
}

static void write_ordered(const job_t *j, int32_t r, int32_t *sel_idx, int32_t sel) {
    int32_t *out = j->out + (int64_t)r * j->k;
    qsort(sel_idx, (size_t)sel, sizeof(int32_t), cmp_asc_i32);
    for (int32_t s = 0; s < j->k; ++s) out[s] = s < sel ? transform(j, r, sel_idx[s]) : -1;
    if (j->ids)
        for (int32_t s = 0; s < j->k; ++s) j->ids[(int64_t)r * j->k + s] = s < sel ? sel_idx[s] : -1;
    j->valid[r] = sel;
}

static void *worker(void *arg) {
    job_t *j = (job_t *)arg;
    for (int32_t r = j->first_row; r < j->rows; r += j->row_step)
        if (one_row(j, r)) { j->status = 1; break; }
    return NULL;
}

/* Rows over `threads` worker threads (<= 1: the calling thread). */
static int run_jobs(job_t *base_in, int32_t threads) {
    job_t base = *base_in;
    const int32_t rows = base.rows;
    if (threads < 1) threads = 1;
    if (threads > rows) threads = rows;
    if (threads == 1) {
        worker(&base);
        return base.status;
    }
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)threads);
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    if (!jobs || !tids) { free(jobs); free(tids); return 1; }
    int32_t started = 0;
    for (int32_t t = 0; t < threads; ++t) {
        jobs[t] = base;
        jobs[t].first_row = t;
        jobs[t].row_step = threads;
        if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0) { jobs[t].status = 1; break; }
        ++started;
    }
    int status = started == threads ? 0 : 1;
    for (int32_t t = 0; t < started; ++t) {
        pthread_join(tids[t], NULL);
        status |= jobs[t].status;
    }
    free(jobs);
    free(tids);
    return status;
}

/*
 * logits: BF16 bits, row r at logits + r * row_stride; valid_len: [rows];
 * block_table: NULL (identity) or [ceil(rows / rows_per_request), table_stride]
 * page ids, page_size elements per page, block_rows physical rows per page;
 * out: [rows, k] int32. threads: worker threads over rows (<= 1: the calling
 * thread only). Returns 0, or 1 on a bad argument or allocation failure.
 */
int oracle_topk_bf16_paged(const uint16_t *logits, int64_t row_stride, int32_t rows,
                           int32_t width, const int32_t *valid_len, int32_t k, int32_t mode,
                           const int32_t *block_table, int32_t table_stride, int32_t page_size,
                           int32_t block_rows, int32_t rows_per_request, int32_t *out,
                           int32_t threads) {
    if (rows < 0 || width < 0 || k < 1 || row_stride < width) return 1;
    if (mode != ORACLE_TOKEN && mode != ORACLE_BLOCK8) return 1;
    if (block_table && (page_size < 1 || block_rows < 1 || rows_per_request < 1)) return 1;
    if (rows == 0) return 0;
    if (!logits || !valid_len || !out) return 1;
    job_t base = {logits, row_stride, rows, width, valid_len, k, mode,
                  block_table, table_stride, page_size, block_rows, rows_per_request,
                  out, 0, 1, 0, 0, NULL, NULL};
    return run_jobs(&base, threads);
}

/* The transform with one table row per row and page_size physical rows per page. */
int oracle_topk_bf16(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                     const int32_t *valid_len, int32_t k, int32_t mode,
                     const int32_t *block_table, int32_t table_stride, int32_t page_size,
                     int32_t *out, int32_t threads) {
    return oracle_topk_bf16_paged(logits, row_stride, rows, width, valid_len, k, mode,
                                  block_table, table_stride, page_size, page_size, 1, out,
                                  threads);
}

/*
 * The ordered variant (token mode): the selection of oracle_topk_bf16_paged in
 * ascending element-index order, -1 past the count; valid: int32 [rows], the
 * counts; ids: NULL or int32 [rows, k], the untransformed indices in the same
 * order, -1 past the count.
 */
int oracle_topk_bf16_ordered(const uint16_t *logits, int64_t row_stride, int32_t rows,
                             int32_t width, const int32_t *valid_len, int32_t k,
                             const int32_t *block_table, int32_t table_stride, int32_t page_size,
                             int32_t block_rows, int32_t rows_per_request, int32_t *out,
                             int32_t *valid, int32_t *ids, int32_t threads) {
    if (rows < 0 || width < 0 || k < 1 || row_stride < width) return 1;
    if (block_table && (page_size < 1 || block_rows < 1 || rows_per_request < 1)) return 1;
    if (rows == 0) return 0;
    if (!logits || !valid_len || !out || !valid) return 1;
    job_t base = {logits, row_stride, rows, width, valid_len, k, ORACLE_TOKEN,
                  block_table, table_stride, page_size, block_rows, rows_per_request,
                  out, 0, 1, 0, 1, valid, ids};
    return run_jobs(&base, threads);
}

/*
 * The scorer's per-8 maxima: tops[r * tops_stride + g] for g < ceil(L / 8) is
 * the largest order key among logits 8g .. 8g + 7 of row r that lie below its
 * valid length L (clamped to [0, width]) and are not NaN, 0 when none is; the
 * entries from ceil(L / 8) to ceil(width / 8) are 0. Returns 0, or 1 on a bad
 * argument.
 */
int oracle_tops(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                const int32_t *valid_len, uint16_t *tops, int64_t tops_stride) {
    if (rows < 0 || width < 0 || row_stride < width) return 1;
    const int32_t groups = (width + 7) / 8;
    if (tops_stride < groups) return 1;
    for (int32_t r = 0; r < rows; ++r) {
        int32_t L = valid_len[r];
        if (L < 0) L = 0;
        if (L > width) L = width;
        const uint16_t *row = logits + (int64_t)r * row_stride;
        for (int32_t g = 0; g < groups; ++g) {
            uint16_t top = 0;
            for (int32_t t = 8 * g; t < 8 * g + 8 && t < L; ++t)
                if (!is_nan_bf16(row[t]) && order_key(row[t]) > top) top = order_key(row[t]);
            tops[(int64_t)r * tops_stride + g] = top;
        }
    }
    return 0;
}

/* One B' word and its plane bit for selected element l at slot j of row r. */
static void put_word(int32_t *orow, int32_t n, int32_t j, int32_t l, uint16_t key) {
    orow[j] = (int32_t)(((uint32_t)key << 16) | (0xFFFFu - ((uint32_t)l & 0xFFFFu)));
    if ((l >> 16) & 1) orow[n + j / 32] |= (int32_t)(1u << (j % 32));
}

/*
 * The words variant (token mode): out int32 [rows, n + n / 32] as described at
 * the top; valid int32 [rows]. n a positive multiple of 32; rows up to 131072
 * elements wide (the plane holds bit 16 of an index). Returns 0, or 1 on a bad
 * argument or allocation failure.
 */
int oracle_topk_bf16_words(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                           const int32_t *valid_len, int32_t n, int32_t *out, int32_t *valid) {
    if (rows < 0 || width < 0 || n < 32 || n % 32 != 0 || row_stride < width || width > (1 << 17))
        return 1;
    if (rows == 0) return 0;
    if (!logits || !valid_len || !out || !valid) return 1;
    const int32_t words = n + n / 32;
    for (int32_t r = 0; r < rows; ++r) {
        const uint16_t *row = logits + (int64_t)r * row_stride;
        int32_t *orow = out + (int64_t)r * words;
        for (int32_t j = 0; j < words; ++j) orow[j] = 0;
        int32_t L = valid_len[r];
        if (L < 0) L = 0;
        if (L > width) L = width;
        if (L <= n) { /* every element, in index order */
            for (int32_t l = 0; l < L; ++l) put_word(orow, n, l, l, order_key(row[l]));
            valid[r] = L;
            continue;
        }
        uint64_t *cand = (uint64_t *)malloc((size_t)L * sizeof(uint64_t));
        if (!cand) return 1;
        int32_t m = 0;
        for (int32_t l = 0; l < L; ++l)
            if (!is_nan_bf16(row[l]))
                cand[m++] = ((uint64_t)order_key(row[l]) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)l);
        qsort(cand, (size_t)m, sizeof(uint64_t), cmp_desc_u64);
        const int32_t sel = m < n ? m : n;
        /* the n-th largest key; with fewer than n candidates every one is "above" */
        const uint16_t T = (uint16_t)(sel == n ? (cand[n - 1] >> 32) : 0);
        int32_t *idx = (int32_t *)malloc((size_t)(sel > 0 ? sel : 1) * sizeof(int32_t));
        if (!idx) { free(cand); return 1; }
        int32_t j = 0;
        for (int pass = 0; pass < 2; ++pass) { /* above T, then ties at T */
            int32_t c = 0;
            for (int32_t s2 = 0; s2 < sel; ++s2) {
                const uint16_t key = (uint16_t)(cand[s2] >> 32);
                if ((pass == 0) == (sel < n || key > T)) idx[c++] = cand_index(cand[s2]);
            }
            qsort(idx, (size_t)c, sizeof(int32_t), cmp_asc_i32);
            for (int32_t t = 0; t < c; ++t) put_word(orow, n, j++, idx[t], order_key(row[idx[t]]));
        }
        valid[r] = sel;
        free(idx);
        free(cand);
    }
    return 0;
}
