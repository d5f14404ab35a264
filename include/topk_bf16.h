/*
 * topk_bf16.h - exact per-row top-k of BF16 logits on GB300 (sm_103a).
 *
 * The operation is the one the vLLM page "decode_topk_cute" states in its module
 * docstring ("What this module computes"): for each row, the indices of its k
 * largest elements, in any order. Exact: every index whose value exceeds the
 * k-th largest, then enough of those equal to it; among elements equal to the
 * k-th largest, the ones with the smallest indices are taken (vLLM kimi_k3
 * "dsa/indexer", IndexerSelect docstring), so the selected set is unique. A row
 * of at most k elements returns 0 .. n-1 and -1 padding without reading its
 * values. Values are compared through the order-preserving 16-bit key of their
 * BF16 bits, x ^ (x < 0 ? 0xFFFF : 0x8000) (sglang PR #39305, Modifications), so
 * -0 ranks below +0 and denormals are ordered by value; NaN elements are never
 * selected. The optional block table is applied as in IndexerSelect.emit of the
 * kimi_k3 indexer page: physical = table[row][i / page] * page + i % page.
 *
 * Every entry point is a plain C function. Pointers named "device" must point to
 * device memory of the current CUDA device; the library never frees, keeps or
 * allocates memory on the caller's behalf and never synchronises the stream.
 * All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 * stream). Calls are thread-safe; the first call on a device sets kernel
 * attributes once.
 *
 * Kernels are launched with programmatic dependent launch where they leave SMs
 * free, and release the next grid on the stream early (unless the hold option
 * is set). A successor launched with programmatic stream serialization may
 * then run alongside the whole call: it must execute griddepcontrol.wait (or
 * cudaGridDependencySynchronize) before it reads any output of this call AND
 * before it writes any input of this call (logits, valid lengths, block table,
 * per-8 maxima), or set hold on this call.
 */
#ifndef TOPK_BF16_H
#define TOPK_BF16_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TOPK_TOKEN = 0,   /* an element is one BF16 logit */
    TOPK_BLOCK8 = 1   /* an element is the NaN-propagating maximum of an aligned
                         group of 8 logits; the row's newest block (the one that
                         holds logit valid_len-1) counts as +inf; a selected block
                         whose value is -inf is written as -1
                         (vLLM decode_topk_cute, module docstring, block mode) */
} topk_mode_t;

typedef enum {
    TOPK_OK = 0,
    TOPK_ERR_ARG = 1,    /* null pointer, rows < 0, bad mode, bad page size or table stride */
    TOPK_ERR_ALIGN = 2,  /* logits not 16-byte aligned, or row_stride not a multiple of 8 */
    TOPK_ERR_K = 3,      /* k outside [1, TOPK_MAX_K] */
    TOPK_ERR_WIDTH = 4,  /* width outside [0, TOPK_MAX_WIDTH], or row_stride < width */
    TOPK_ERR_CUDA = 5,   /* a CUDA call failed (launch or attribute); see cudaGetLastError */
    TOPK_ERR_SIZE = 6    /* topk_bf16_select_static: more rows than its table holds, or rows
                            wider than one 16384-logit stage */
} topk_status_t;

#define TOPK_MAX_K 2048
#define TOPK_MAX_WIDTH (1 << 20)
#define TOPK_STATIC_MAX_ROWS 65536   /* rows per call of topk_bf16_select_static */
#define TOPK_STATIC_MAX_WIDTH 16384  /* logits per row of topk_bf16_select_static */

/*
 * Exact top-k of every row (the operation described at the top of this file).
 *
 * logits       device, BF16 bit patterns; row r starts at logits + r * row_stride.
 *              The base must be 16-byte aligned and row_stride a multiple of 8, so
 *              that every row is read as whole 16-byte vectors. The buffer must be
 *              readable for rows * row_stride elements.
 * row_stride   elements between consecutive rows (>= width).
 * rows         number of rows (0 is a no-op that returns TOPK_OK).
 * width        logits per row that may be valid, 0 .. TOPK_MAX_WIDTH.
 * valid_len    device, int32 [rows]: valid logits of each row (a prefix); values
 *              outside [0, width] are clamped on the device. n = valid_len in token
 *              mode, ceil(valid_len / 8) in block mode.
 * k            1 .. TOPK_MAX_K.
 * mode         TOPK_TOKEN or TOPK_BLOCK8.
 * block_table  NULL for logical indices, else device int32 [rows, table_stride]:
 *              row r's page ids; selected element i is written as
 *              block_table[r * table_stride + i / page_size] * page_size + i % page_size.
 *              table_stride must be >= ceil(width_elements / page_size), where
 *              width_elements is width (token) or ceil(width / 8) (block).
 * page_size    elements per page, a power of two (64 in the pages' layout); ignored
 *              when block_table is NULL.
 * out          device, int32 [rows, k], fully written: the selected (transformed)
 *              indices in any order, then -1 for the remaining slots. Must not
 *              overlap the inputs.
 * stream       cudaStream_t to enqueue on.
 *
 * Returns TOPK_OK once the work is enqueued, or an error status without
 * enqueueing anything. Device-side data is never validated by trapping.
 */
topk_status_t topk_bf16_select(const uint16_t *logits, int64_t row_stride, int32_t rows,
                               int32_t width, const int32_t *valid_len, int32_t k,
                               topk_mode_t mode, const int32_t *block_table,
                               int32_t table_stride, int32_t page_size, int32_t *out,
                               void *stream);

/*
 * topk_bf16_select with the full block-table transform of the indexer page
 * (vLLM kimi_k3 "dsa/indexer": IndexerSelect's docstring and kernel, and
 * IndexerSelect.emit): rows come in requests of rows_per_request consecutive rows
 * that share one table row (request = row / rows_per_request), and each page of
 * page_size elements maps to block_rows physical rows:
 *     physical = block_table[request * table_stride + i / page_size] * block_rows
 *                + i % page_size.
 * block_rows is a power of two >= page_size (64, or e.g. 2048 in hybrid models);
 * the caller keeps page ids small enough that physical indices fit int32.
 * block_table holds ceil(rows / rows_per_request) rows. topk_bf16_select is this
 * call with rows_per_request = 1 and block_rows = page_size.
 * Errors as topk_bf16_select, plus TOPK_ERR_ARG for rows_per_request < 1 or a bad
 * block_rows (checked when block_table is not NULL).
 */
topk_status_t topk_bf16_select_paged(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                     int32_t width, const int32_t *valid_len, int32_t k,
                                     topk_mode_t mode, const int32_t *block_table,
                                     int32_t table_stride, int32_t page_size, int32_t block_rows,
                                     int32_t rows_per_request, int32_t *out, void *stream);

/* Human-readable name of a status (a static string). */
const char *topk_bf16_status_string(topk_status_t status);

/*
 * Options for topk_bf16_select_ex (and the ordered select and B' words): test
 * and diagnosis hooks, which change which internal path computes the result,
 * never the result itself, and the hold flag, which changes only when the next
 * kernel on the stream may start. Zero-initialise the whole struct.
 */
typedef struct {
    int32_t force_direct;   /* 1: skip the group-representative cutoff; every first
                               tile takes the exact whole-tile radix path (the fallback) */
    int32_t cluster;        /* 0: automatic; else CTAs per row: 1, 2, 4, 8 or 16 */
    uint32_t *counters;     /* NULL, or device uint32 [TOPK_NUM_COUNTERS] that each
                               launch adds its path counts and cycle split to */
    int32_t path;           /* rows wider than one stage: 0 automatic, 1 candidate buffer
                               (streamed), 2 resident keys (direct; rows whose cluster
                               shares fit 16384 keys per CTA) */
    int32_t hold;           /* 0: the kernel lets the next kernel on the stream start early
                               (programmatic dependent launch; that kernel must wait for this
                               grid before it reads the output and before it writes any of
                               this call's inputs). Nonzero: it does not, so a next kernel
                               launched that way starts only once this grid has completed:
                               for consumers that read the output, or producers that write
                               the next step's inputs, before their wait (the indexer page,
                               IndexerSelect's release flag). */
} topk_bf16_options_t;

/* Indices into topk_bf16_options_t.counters. */
enum {
    TOPK_CNT_BYPASS_ROWS = 0,    /* rows with n <= k */
    TOPK_CNT_TILE_SAMPLED = 1,   /* first tiles (and resident-keys rows) cut by the k-th largest
                                    group representative */
    TOPK_CNT_TILE_EXACT = 2,     /* first tiles (and resident-keys rows) cut by the exact path
                                    (every key its own representative): forced, fallen back to,
                                    or rows too short for groups */
    TOPK_CNT_TILE_UNBOUNDED = 3, /* fewer than k usable representatives: exact path taken */
    TOPK_CNT_TILE_OVERFLOW = 4,  /* more survivors than buffer room (resident-keys rows: the
                                    k-th key past the cut's window): exact path taken */
    TOPK_CNT_TILE_TAKE_ALL = 5,  /* first tiles with at most k candidates */
    TOPK_CNT_COMPACTIONS = 6,    /* candidate-buffer compactions */
    TOPK_CNT_REFILLS = 7,        /* tiles that filled the buffer and resumed after a compaction */
    TOPK_CNT_CLUSTER_MERGES = 8, /* rows merged across a cluster of CTAs */
    TOPK_CNT_ROUNDS = 9,         /* tiles streamed in total */
    /* SM clock cycles thread 0 of each CTA spent, summed over CTAs: */
    TOPK_CNT_CYC_WAIT = 10,      /* waiting for a stage */
    TOPK_CNT_CYC_SELECT = 11,    /* first-tile selects */
    TOPK_CNT_CYC_FILTER = 12,    /* later tiles (compactions included) */
    TOPK_CNT_CYC_FINISH = 13,    /* the row's final select, merge and write */
    TOPK_CNT_CYC_COMPACT = 14,   /* buffer compactions */
    TOPK_CNT_CYC_REPS = 15,      /* first-tile select, split: representatives histogram */
    TOPK_CNT_CYC_CUT = 16,       /*   the representatives' cut */
    TOPK_CNT_CYC_SURVIVORS = 17, /*   the survivor pass */
    TOPK_CNT_CYC_EXACT = 18,     /*   the exact cut among survivors and the tie appends */
    TOPK_CNT_GUESS_HIT = 19,     /* rows cut by a carried-over cut: one-tile rows by the cut of
                                    the CTA's previous row, resident-keys and streamed rows by
                                    the k-th key of the cluster's previous row less a margin
                                    (checked by the exact survivor counts, the window sums or
                                    the buffers' final counts) */
    TOPK_CNT_GUESS_MISS = 20,    /* carried-over cuts dropped: fewer than k keys at or above
                                    it, more survivors than buffer room, (resident-keys rows)
                                    the k-th key past the cut's window, or (streamed rows) a
                                    first tile whose count above it, scaled to the row, is
                                    below k or above 8k, or a row streamed again after ending
                                    with fewer than k keys above it */
    /* streamed rows, later tiles, split (thread 0 of each CTA): */
    TOPK_CNT_CYC_F_PREP = 21,    /*   threshold update, compaction, running-histogram rebuild */
    TOPK_CNT_CYC_F_QUEUE = 22,   /*   candidate-vector queue */
    TOPK_CNT_CYC_F_APPEND = 23,  /*   appends to the buffer */
    TOPK_CNT_CYC_F_SYNC = 24,    /*   the tile's barrier (and any refill) */
    TOPK_CNT_CYC_F_FIND = 25,    /*   the buffer's k-th key for the next threshold */
    TOPK_CNT_CYC_F_LOOP = 26,    /*   end of tile: barrier and the next copy's issue */
    TOPK_CNT_TIE_FILLS = 27,     /* streamed first tiles completed with lowest-index ties at their cut */
    TOPK_CNT_DIRECT_ROWS = 28,   /* rows selected from resident keys (the direct kernel) */
    TOPK_CNT_CYC_KERNEL = 29,    /* resident-keys kernel: entry to exit (thread 0 of each CTA) */
    TOPK_CNT_CYC_ALIGN = 30,     /* resident-keys rows: the first cluster-wide sum after the
                                    share is in (mostly waiting for the cluster's slowest CTA) */
    TOPK_CNT_ORDERED_TOPS = 31,  /* ordered rows selected from the tops' bound */
    TOPK_CNT_ORDERED_EXACT = 32, /* ordered rows that took the exact select over every key */
    TOPK_NUM_COUNTERS = 40
};

/* topk_bf16_select with options (NULL = defaults). Same arguments and errors,
   plus TOPK_ERR_ARG for an unsupported cluster size. */
topk_status_t topk_bf16_select_ex(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                  int32_t width, const int32_t *valid_len, int32_t k,
                                  topk_mode_t mode, const int32_t *block_table,
                                  int32_t table_stride, int32_t page_size, int32_t *out,
                                  void *stream, const topk_bf16_options_t *options);

/*
 * topk_bf16_select_static: the same selection as topk_bf16_select, for rows of
 * at most TOPK_STATIC_MAX_WIDTH logits (one 32 KiB stage), where each row
 * starts from the cut that worked for the same row index in the previous call.
 * No source page has a counterpart. A per-row table like this is scratch that
 * would normally be a buffer the caller allocates and passes in; this entry
 * point serves callers that cannot allocate device memory at all (code running
 * inside a stream capture that must not record allocations, programs under a
 * fixed device-memory budget with no allocator, plug-ins whose host owns every
 * allocation). The table lives in the library itself: TOPK_STATIC_MAX_ROWS
 * 32-bit words (256 KiB) in a static array of every device that loads the
 * library, held until the process exits; the call allocates nothing and the
 * caller passes only inputs and outputs, as for topk_bf16_select.
 *
 * The table holds per-row starting cuts for decode loops, where row r of one
 * call is the same request as row r of the last: a starting cut is checked by
 * an exact count like any other and dropped when it does not hold, so results
 * are always exact. Every call on a device shares the table and leaves its own
 * cuts in it; nothing needs clearing, and calls that overlap on the GPU (other
 * streams) race on it harmlessly (any entry is a valid starting point).
 *
 * The first call on a device takes the table's device address and sets the
 * kernels' attributes (once per device, with that device current): make that
 * first call before capturing a stream into a CUDA graph.
 *
 * Arguments and outputs as topk_bf16_select. Errors as topk_bf16_select, plus
 * TOPK_ERR_SIZE for rows > TOPK_STATIC_MAX_ROWS or width > TOPK_STATIC_MAX_WIDTH.
 */
topk_status_t topk_bf16_select_static(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                      int32_t width, const int32_t *valid_len, int32_t k,
                                      topk_mode_t mode, const int32_t *block_table,
                                      int32_t table_stride, int32_t page_size, int32_t *out,
                                      void *stream);

/*
 * The ordered select of the indexer page (vLLM kimi_k3 "dsa/indexer":
 * IndexerSelect's docstring, kernel and write_selected), token mode: the same
 * selected set as topk_bf16_select_paged, written in ascending element-index
 * order ("key order": the page's keys are token positions), bounded by the
 * scorer's per-8 maxima so that only the vectors that can hold a selected key
 * are read.
 *
 * tops         NULL, or device uint16 [rows, tops_stride], 16-byte aligned:
 *              tops[r * tops_stride + g], for g < ceil(valid_len[r] / 8), is the
 *              largest order key x ^ (x < 0 ? 0xFFFF : 0x8000) among logits
 *              8g .. 8g + 7 of row r that lie below its valid length and are not
 *              NaN, 0 when there is none (what IndexerScore.rows_out writes for
 *              the select). They must be exactly that: a row is read only where
 *              its tops reach the row's bound (wrong tops give a wrong result,
 *              never an out-of-bounds access). NULL: every row takes the exact
 *              select over all of its logits.
 * tops_stride  a multiple of 8, at least ceil(ceil(width / 8) / 8) * 8 (whole
 *              16-byte pieces of tops are read; entries past a row's valid
 *              groups are ignored).
 * out          device int32 [rows, k]: the selected indices in ascending index
 *              order, transformed as in topk_bf16_select_paged, then -1.
 * valid        device int32 [rows]: each row's count of selected indices: n
 *              when n <= k (the row is taken whole without reading values, as
 *              in topk_bf16_select), else k, or the row's non-NaN elements when
 *              they are fewer.
 * ids          NULL, or device int32 [rows, k]: the untransformed indices in the
 *              same order, then -1.
 * options      NULL, or test hooks: counters (TOPK_CNT_BYPASS_ROWS,
 *              TOPK_CNT_ORDERED_TOPS, TOPK_CNT_ORDERED_EXACT), force_direct
 *              (tops ignored: the exact select on every row). Other fields unused.
 * The remaining arguments are those of topk_bf16_select_paged (mode is token).
 * Errors as topk_bf16_select_paged, plus TOPK_ERR_ARG for a NULL valid or a
 * short tops_stride and TOPK_ERR_ALIGN for misaligned tops, tops_stride, valid
 * or ids.
 */
topk_status_t topk_bf16_select_ordered(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                       int32_t width, const int32_t *valid_len, int32_t k,
                                       const uint16_t *tops, int64_t tops_stride,
                                       const int32_t *block_table, int32_t table_stride,
                                       int32_t page_size, int32_t block_rows, int32_t rows_per_request,
                                       int32_t *out, int32_t *valid, int32_t *ids, void *stream,
                                       const topk_bf16_options_t *options);

/*
 * The local top-n of token rows as the DCP merge's B' words (vLLM kimi_k3
 * "dsa/indexer": IndexerLocalTopk's docstring, kernel and candidate), one GPU's
 * part: out[r * (n + n / 32) + j], j < n, is (key << 16) | (0xFFFF - (l & 0xFFFF))
 * for the j-th selected element l of row r, with key = x ^ (x < 0 ? 0xFFFF :
 * 0x8000) of its BF16 bits, or 0 for an empty slot; bit j % 32 of
 * out[r * (n + n / 32) + n + j / 32] is bit 16 of l. Order: the selected
 * elements whose key exceeds the row's n-th largest key, in index order, then
 * the ties at it that are taken (the lowest indices), in index order. A row of at
 * most n elements takes every one of them, in index order (their words hold
 * their keys, whatever the values); in longer rows NaN is never selected, and
 * when fewer than n are eligible all of them are taken, in index order.
 * valid[r]: the count. The selection is the one topk_bf16_select makes.
 *
 * n            32 .. TOPK_MAX_K, a multiple of 32.
 * width        0 .. 131072 (the plane holds bit 16 of an index).
 * tops         NULL, or the per-8 maxima as for topk_bf16_select_ordered (the
 *              bound that limits the vectors read); NULL: the exact select.
 * out          device int32 [rows, n + n / 32]; valid: device int32 [rows].
 * options      NULL, or test hooks as for topk_bf16_select_ordered.
 * logits, row_stride, rows, valid_len, stream as in topk_bf16_select. Errors as
 * topk_bf16_select_ordered, plus TOPK_ERR_ARG for n not a multiple of 32 or a
 * width above 131072.
 */
topk_status_t topk_bf16_select_words(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                     int32_t width, const int32_t *valid_len, int32_t n,
                                     const uint16_t *tops, int64_t tops_stride, int32_t *out,
                                     int32_t *valid, void *stream, const topk_bf16_options_t *options);

/*
 * The per-8 maxima topk_bf16_select_ordered is bounded by, for producers that
 * do not write them (IndexerScore.rows_out on the indexer page writes them
 * with the logits): tops[r * tops_stride + g] = the largest order key among
 * logits 8g .. 8g + 7 of row r below valid_len[r] (clamped to [0, width]) that
 * are not NaN, 0 when there is none, for every g < ceil(ceil(width / 8) / 8) * 8.
 * logits, row_stride, rows, width, valid_len as in topk_bf16_select; tops:
 * device uint16, 16-byte aligned; tops_stride: a multiple of 8, at least
 * ceil(ceil(width / 8) / 8) * 8. Errors as topk_bf16_select for those
 * arguments, TOPK_ERR_ALIGN for a misaligned tops or tops_stride, TOPK_ERR_ARG
 * for a short tops_stride.
 */
topk_status_t topk_bf16_tops(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                             const int32_t *valid_len, uint16_t *tops, int64_t tops_stride,
                             void *stream);

/*
 * The launch topk_bf16_select would make for these sizes on the current device:
 * CTAs per row, threads per CTA, dynamic shared memory bytes, the kernel
 * variant (0 = one-tile rows, 1 = streamed rows, 2 = resident keys) and the CTAs
 * launched (persistent: at most what is resident at once; rows beyond that are
 * taken in turn). Any output pointer may be NULL.
 */
topk_status_t topk_bf16_plan(int32_t rows, int32_t width, int32_t k, topk_mode_t mode,
                             int32_t *cluster, int32_t *threads, int32_t *smem_bytes,
                             int32_t *variant, int32_t *ctas);

/*
 * Device-side status word of the current device: nonzero bits record a bounded
 * wait that gave up (bit 0), an internal capacity or range check that failed
 * (bit 1), or, in a library built with -DTOPK_DEBUG, a shared-memory index out
 * of range (bit 2, the access skipped); none happens in correct operation, and
 * the kernels never trap.
 * Synchronises the device. clear != 0 resets the word afterwards.
 */
topk_status_t topk_bf16_device_status(uint32_t *flags, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* TOPK_BF16_H */
