// Host side of the library: argument checks, the launch plan (which kernel,
// cluster size and grid for a call), the launches, and the C ABI declared in
// topk_bf16.h.

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <initializer_list>
#include <mutex>

#include "params.h"
#include "topk_bf16.h"

namespace topk {

// ------------------------------------------------------------------ host side

struct DeviceInit {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int sms = 0;
    int per_sm[2][2] = {{0, 0}, {0, 0}};   // resident CTAs per SM, [block][wide]
    int per_sm_one[2][ONE_BUILDS] = {};    // the one-tile kernel, [block][build]
    int per_sm_direct[2] = {0, 0};         // the resident-keys kernel, [block]
    // Clusters of 1, 2, 4, 8, 16 CTAs resident at once, [direct][block][log2 size]
    // (a cluster's CTAs share one GPC, so this can be less than the slots / size).
    int cap[2][2][5] = {};
};

// Clusters of c CTAs of this kernel that fit on the device at once; 0 if none
// (or if the runtime cannot say, e.g. a size above what the kernel allows).
int cluster_capacity(const Variant &v, int threads, int c) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(v.smem);
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = static_cast<unsigned>(c);
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    cfg.attrs = &a;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, v.fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}
DeviceInit g_init[64];

cudaError_t init_device(int dev, DeviceInit *&out) {
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DeviceInit &d = g_init[dev];
    std::call_once(d.once, [&]() {
        cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        for (int b = 0; b < 2 && e == cudaSuccess; ++b)
            for (int w = 1; w < 2 && e == cudaSuccess; ++w) {
                const Variant v = stream_variant(b != 0);
                e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem);
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e == cudaSuccess)
                    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.per_sm[b][w], v.fn, THREADS,
                                                                      static_cast<size_t>(v.smem));
                if (e == cudaSuccess && d.per_sm[b][w] < 1) e = cudaErrorInvalidConfiguration;
            }
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            const Variant v = direct_variant(b != 0);
            e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.per_sm_direct[b], v.fn, direct::NT,
                                                                  static_cast<size_t>(v.smem));
            if (e == cudaSuccess && d.per_sm_direct[b] < 1) e = cudaErrorInvalidConfiguration;
        }
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ordered_variant().fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     ordered_variant().smem);
        for (int b = 0; b < 2 && e == cudaSuccess; ++b)
            for (int l = 0; l < 5; ++l) {
                const int c = 1 << l;
                d.cap[0][b][l] = l == 0 ? d.sms * d.per_sm[b][1] : cluster_capacity(stream_variant(b != 0), THREADS, c);
                d.cap[1][b][l] = l == 0 ? d.sms * d.per_sm_direct[b]
                                        : cluster_capacity(direct_variant(b != 0), direct::NT, c);
            }
        for (int b = 0; b < 2 && e == cudaSuccess; ++b)
            for (int w = 0; w < ONE_BUILDS && e == cudaSuccess; ++w) {
                const Variant v = one_variant(b != 0, w);
                e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem);
                if (e == cudaSuccess)
                    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.per_sm_one[b][w], v.fn, one_threads(w),
                                                                      static_cast<size_t>(v.smem));
                if (e == cudaSuccess && d.per_sm_one[b][w] < 1) e = cudaErrorInvalidConfiguration;
            }
        d.err = e;
    });
    out = &d;
    return d.err;
}

enum Kind { KIND_ONE = 0, KIND_STREAM = 1, KIND_DIRECT = 2 };

struct Plan {
    int kind;          // which kernel
    int cluster;
    int build;         // one-tile rows: which build (see one_variant)
    int threads;
    int64_t clusters;  // persistent clusters launched
    bool spare;        // some resident slots stay free (the launch may overlap the previous one)
};

// One CTA per row when a row fits one stage. Wider rows: block rows keep
// their keys resident across the smallest cluster that holds them (the
// direct kernel); token rows stream through a candidate buffer. Either way the
// cluster grows, up to 16, while that puts about one CTA on every resident slot,
// keeps every row's cluster resident at once and leaves every CTA at least one
// stage. Clusters are persistent, so the grid never exceeds what is resident at
// once (clusters are placed whole, within one GPC: the runtime's count of
// resident clusters, not the slots / size). path: 0 automatic, 1 streamed, 2 direct.
Plan make_plan(int rows, int width, int k, const DeviceInit &d, bool block, int forced, int path) {
    const int64_t vecs = (static_cast<int64_t>(width) + 7) / 8;
    const int64_t per_vec = block ? 1 : 8;  // elements per vector
    Plan pl{KIND_ONE, 1, 0, THREADS, 1, false};
    int c_res = 1;  // the smallest cluster whose shares fit as resident keys
    while (c_res < 16 && (vecs + c_res - 1) / c_res * per_vec > direct::RES) c_res *= 2;
    const bool fits = (vecs + c_res - 1) / c_res * per_vec <= direct::RES;
    if (path == 2 && fits) pl.kind = KIND_DIRECT;
    else if (path == 1 || vecs > TILE_VEC || forced > 1) pl.kind = block && fits && path != 1 ? KIND_DIRECT : KIND_STREAM;
    if (pl.kind == KIND_ONE) {
        // Rows that leave SMs idle at one 512-thread CTA each take that build:
        // twice the threads on every row, so half the row's latency.
        pl.build = rows <= d.sms * d.per_sm_one[block][2] ? 2 : (k <= 1024 ? 0 : 1);
        pl.threads = one_threads(pl.build);
    }
    const int per_sm = pl.kind == KIND_ONE ? d.per_sm_one[block][pl.build]
                       : pl.kind == KIND_STREAM ? d.per_sm[block][1] : d.per_sm_direct[block];
    const int64_t slots = static_cast<int64_t>(d.sms) * per_sm;
    auto resident = [&](int c) -> int64_t {
        if (pl.kind == KIND_ONE) return slots;
        int l = 0;
        while ((1 << l) < c) ++l;
        const int n = d.cap[pl.kind == KIND_DIRECT][block][l];
        return n > 0 ? n : slots / c;
    };
    if (forced > 0) {
        pl.cluster = pl.kind == KIND_DIRECT ? max(forced, c_res) : forced;
    } else if (pl.kind != KIND_ONE) {
        const int64_t stages = (vecs + TILE_VEC - 1) / TILE_VEC;
        int c = pl.kind == KIND_DIRECT ? c_res : 1;
        while (c < 16 && static_cast<int64_t>(rows) * c * 5 < slots * 4 && 2 * c <= stages &&
               rows <= resident(2 * c))
            c *= 2;
        pl.cluster = c;
    }
    const int64_t max_clusters = resident(pl.cluster) > 0 ? resident(pl.cluster) : 1;
    pl.clusters = rows < max_clusters ? rows : max_clusters;
    pl.spare = pl.clusters * pl.cluster < slots;
    return pl;
}

topk_status_t check_args(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                         const int32_t *valid_len, int32_t k, topk_mode_t mode,
                         const int32_t *table, int32_t table_stride, int32_t page_size,
                         const int32_t *out) {
    if (rows < 0) return TOPK_ERR_ARG;
    if (mode != TOPK_TOKEN && mode != TOPK_BLOCK8) return TOPK_ERR_ARG;
    if (k < 1 || k > TOPK_MAX_K) return TOPK_ERR_K;
    if (width < 0 || width > TOPK_MAX_WIDTH || row_stride < width) return TOPK_ERR_WIDTH;
    if (rows == 0) return TOPK_OK;
    if (!logits || !valid_len || !out) return TOPK_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(logits) & 15u) != 0 || (row_stride & 7) != 0) return TOPK_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(out) & 3u) != 0 || (reinterpret_cast<uintptr_t>(valid_len) & 3u) != 0)
        return TOPK_ERR_ALIGN;
    if (table) {
        if (page_size < 1 || (page_size & (page_size - 1)) != 0) return TOPK_ERR_ARG;
        const int64_t elems = mode == TOPK_BLOCK8 ? (static_cast<int64_t>(width) + 7) / 8 : width;
        if (table_stride < (elems + page_size - 1) / page_size) return TOPK_ERR_ARG;
        if ((reinterpret_cast<uintptr_t>(table) & 3u) != 0) return TOPK_ERR_ALIGN;
    }
    return TOPK_OK;
}

topk_status_t launch(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                     const int32_t *valid_len, int32_t k, topk_mode_t mode, const int32_t *table,
                     int32_t table_stride, int32_t page_size, int32_t block_rows, int32_t q,
                     int32_t *out, void *stream, const topk_bf16_options_t *opt) {
    if (q < 1) return TOPK_ERR_ARG;
    if (table && (block_rows < page_size || (block_rows & (block_rows - 1)) != 0)) return TOPK_ERR_ARG;
    topk_status_t st = check_args(logits, row_stride, rows, width, valid_len, k, mode, table,
                                  table_stride, page_size, out);
    if (st != TOPK_OK || rows == 0) return st;
    const int forced = opt ? opt->cluster : 0;
    const int path = opt ? opt->path : 0;
    if (path < 0 || path > 2) return TOPK_ERR_ARG;
    if (forced != 0 && forced != 1 && forced != 2 && forced != 4 && forced != 8 && forced != 16)
        return TOPK_ERR_ARG;
    int dev = 0;
    DeviceInit *d = nullptr;
    if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (init_device(dev, d) != cudaSuccess) return TOPK_ERR_CUDA;

    const bool block = mode == TOPK_BLOCK8;
    const Plan pl = make_plan(rows, width, k, *d, block, forced, path);
    const Variant v = pl.kind == KIND_ONE ? one_variant(block, pl.build)
                      : pl.kind == KIND_STREAM ? stream_variant(block) : direct_variant(block);
    const int threads = pl.threads;

    Params prm;
    prm.logits = logits;
    prm.row_stride = row_stride;
    prm.rows = rows;
    prm.width = width;
    prm.valid_len = valid_len;
    prm.k = k;
    prm.table = table;
    prm.table_stride = table_stride;
    prm.block_rows = block_rows;
    prm.rows_per_request = q;
    prm.page_shift = 0;
    if (table)
        while ((1 << prm.page_shift) < page_size) ++prm.page_shift;
    prm.out = out;
    prm.counters = opt ? opt->counters : nullptr;
    prm.force_direct = opt ? opt->force_direct : 0;
    prm.release = (opt && opt->hold) ? 0 : 1;

    const int64_t blocks = pl.clusters * pl.cluster;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(v.smem);
    cfg.stream = static_cast<cudaStream_t>(stream);
    // A grid that leaves resident slots free may start while the previous
    // kernel on the stream finishes (see grid_dependency_wait); one that fills
    // every slot would only crowd the previous one's tail.
    cudaLaunchAttribute attr[2];
    unsigned n_attr = 0;
    if (pl.spare) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr++].val.programmaticStreamSerializationAllowed = 1;
    }
    if (pl.cluster > 1) {  // a lone CTA per row needs no cluster
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = static_cast<unsigned>(pl.cluster);
        attr[n_attr].val.clusterDim.y = 1;
        attr[n_attr++].val.clusterDim.z = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    void *args[] = {&prm};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, v.fn, args);
    return e == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}

// topk_bf16_select_static: the one-tile kernel with per-row starting cuts in
// the library's static table (no allocation anywhere on this path).
topk_status_t launch_static(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                            const int32_t *valid_len, int32_t k, topk_mode_t mode, const int32_t *table,
                            int32_t table_stride, int32_t page_size, int32_t *out, void *stream) {
    topk_status_t st = check_args(logits, row_stride, rows, width, valid_len, k, mode, table, table_stride,
                                  page_size, out);
    if (st != TOPK_OK) return st;
    if (rows > TOPK_STATIC_MAX_ROWS || width > TOPK_STATIC_MAX_WIDTH) return TOPK_ERR_SIZE;
    if (rows == 0) return TOPK_OK;
    int dev = 0;
    DeviceInit *d = nullptr;
    if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (init_device(dev, d) != cudaSuccess) return TOPK_ERR_CUDA;
    uint32_t *row_carry = nullptr;
    if (static_row_carry(dev, &row_carry) != cudaSuccess || row_carry == nullptr) return TOPK_ERR_CUDA;

    const bool block = mode == TOPK_BLOCK8;
    const Plan pl = make_plan(rows, width, k, *d, block, 0, 0);
    if (pl.kind != KIND_ONE) return TOPK_ERR_SIZE;  // (cannot happen within the width limit)
    const Variant v = one_static_variant(block, pl.build);

    Params prm;
    prm.logits = logits;
    prm.row_stride = row_stride;
    prm.rows = rows;
    prm.width = width;
    prm.valid_len = valid_len;
    prm.k = k;
    prm.table = table;
    prm.table_stride = table_stride;
    prm.block_rows = page_size;
    prm.rows_per_request = 1;
    prm.page_shift = 0;
    if (table)
        while ((1 << prm.page_shift) < page_size) ++prm.page_shift;
    prm.out = out;
    prm.counters = nullptr;
    prm.force_direct = 0;
    prm.release = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.clusters), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(pl.threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(v.smem);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    unsigned n_attr = 0;
    if (pl.spare) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr++].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    void *args[] = {&prm, &row_carry};
    return cudaLaunchKernelExC(&cfg, v.fn, args) == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}

// The ordered select: one CTA per row, as many rows at once as there are SMs.
topk_status_t launch_ordered(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                             const int32_t *valid_len, int32_t k, const uint16_t *tops,
                             int64_t tops_stride, const int32_t *table, int32_t table_stride,
                             int32_t page_size, int32_t block_rows, int32_t q, int32_t *out,
                             int32_t *valid, int32_t *ids, void *stream,
                             const topk_bf16_options_t *opt, bool words = false) {
    if (q < 1) return TOPK_ERR_ARG;
    if (words && (k % 32 != 0 || width > (1 << 17) || table || ids)) return TOPK_ERR_ARG;
    if (table && (block_rows < page_size || (block_rows & (block_rows - 1)) != 0)) return TOPK_ERR_ARG;
    topk_status_t st = check_args(logits, row_stride, rows, width, valid_len, k, TOPK_TOKEN, table,
                                  table_stride, page_size, out);
    if (st != TOPK_OK || rows == 0) return st;
    if (!valid) return TOPK_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(valid) & 3u) != 0 || (reinterpret_cast<uintptr_t>(ids) & 3u) != 0)
        return TOPK_ERR_ALIGN;
    if (tops) {
        const int64_t groups = (static_cast<int64_t>(width) + 7) / 8;
        if ((reinterpret_cast<uintptr_t>(tops) & 15u) != 0 || (tops_stride & 7) != 0) return TOPK_ERR_ALIGN;
        if (tops_stride < (groups + 7) / 8 * 8) return TOPK_ERR_ARG;
    }
    int dev = 0;
    DeviceInit *d = nullptr;
    if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (init_device(dev, d) != cudaSuccess) return TOPK_ERR_CUDA;

    ordered::OParams prm;
    prm.logits = logits;
    prm.row_stride = row_stride;
    prm.rows = rows;
    prm.width = width;
    prm.valid_len = valid_len;
    prm.k = k;
    prm.tops = (opt && opt->force_direct) ? nullptr : tops;
    prm.tops_stride = tops_stride;
    prm.table = table;
    prm.table_stride = table_stride;
    prm.page_shift = 0;
    if (table)
        while ((1 << prm.page_shift) < page_size) ++prm.page_shift;
    prm.block_rows = block_rows;
    prm.rows_per_request = q;
    prm.out = out;
    prm.valid = valid;
    prm.ids = ids;
    prm.counters = opt ? opt->counters : nullptr;
    prm.words = words ? 1 : 0;
    prm.release = (opt && opt->hold) ? 0 : 1;

    const int grid = rows < d->sms ? rows : d->sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(ordered::NT, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(ordered_variant().smem);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    unsigned n_attr = 0;
    if (grid < d->sms) {  // SMs left free: the launch may overlap the previous kernel's tail
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr++].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    void *args[] = {&prm};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, ordered_variant().fn, args);
    return e == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}

}  // namespace topk

extern "C" {

topk_status_t topk_bf16_tops(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                             const int32_t *valid_len, uint16_t *tops, int64_t tops_stride,
                             void *stream) {
    topk_status_t st = topk::check_args(logits, row_stride, rows, width, valid_len, 1, TOPK_TOKEN,
                                        nullptr, 0, 0, reinterpret_cast<const int32_t *>(tops));
    if (st != TOPK_OK || rows == 0) return st;
    const int64_t groups = (static_cast<int64_t>(width) + 7) / 8;
    const int64_t pieces = (groups + 7) / 8;
    if ((reinterpret_cast<uintptr_t>(tops) & 15u) != 0 || (tops_stride & 7) != 0) return TOPK_ERR_ALIGN;
    if (tops_stride < pieces * 8) return TOPK_ERR_ARG;
    if (pieces == 0) return TOPK_OK;
    int dev = 0;
    topk::DeviceInit *d = nullptr;
    if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (topk::init_device(dev, d) != cudaSuccess) return TOPK_ERR_CUDA;
    const int64_t total = static_cast<int64_t>(rows) * pieces;
    const int64_t want = (total + 255) / 256;
    const unsigned blocks = static_cast<unsigned>(want < 8LL * d->sms ? want : 8LL * d->sms);
    return topk::launch_tops(logits, row_stride, rows, width, valid_len, tops, tops_stride,
                             static_cast<int32_t>(pieces), blocks, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? TOPK_OK
               : TOPK_ERR_CUDA;
}

topk_status_t topk_bf16_select_words(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                     int32_t width, const int32_t *valid_len, int32_t n,
                                     const uint16_t *tops, int64_t tops_stride, int32_t *out,
                                     int32_t *valid, void *stream, const topk_bf16_options_t *options) {
    return topk::launch_ordered(logits, row_stride, rows, width, valid_len, n, tops, tops_stride,
                                nullptr, 0, 64, 64, 1, out, valid, nullptr, stream, options, true);
}

topk_status_t topk_bf16_select_ordered(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                       int32_t width, const int32_t *valid_len, int32_t k,
                                       const uint16_t *tops, int64_t tops_stride,
                                       const int32_t *block_table, int32_t table_stride,
                                       int32_t page_size, int32_t block_rows, int32_t rows_per_request,
                                       int32_t *out, int32_t *valid, int32_t *ids, void *stream,
                                       const topk_bf16_options_t *options) {
    return topk::launch_ordered(logits, row_stride, rows, width, valid_len, k, tops, tops_stride,
                                block_table, table_stride, page_size, block_rows, rows_per_request,
                                out, valid, ids, stream, options);
}

topk_status_t topk_bf16_select(const uint16_t *logits, int64_t row_stride, int32_t rows,
                               int32_t width, const int32_t *valid_len, int32_t k,
                               topk_mode_t mode, const int32_t *block_table,
                               int32_t table_stride, int32_t page_size, int32_t *out,
                               void *stream) {
    return topk::launch(logits, row_stride, rows, width, valid_len, k, mode, block_table,
                        table_stride, page_size, page_size, 1, out, stream, nullptr);
}

topk_status_t topk_bf16_select_paged(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                     int32_t width, const int32_t *valid_len, int32_t k,
                                     topk_mode_t mode, const int32_t *block_table,
                                     int32_t table_stride, int32_t page_size, int32_t block_rows,
                                     int32_t rows_per_request, int32_t *out, void *stream) {
    return topk::launch(logits, row_stride, rows, width, valid_len, k, mode, block_table,
                        table_stride, page_size, block_rows, rows_per_request, out, stream, nullptr);
}

topk_status_t topk_bf16_select_static(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                      int32_t width, const int32_t *valid_len, int32_t k,
                                      topk_mode_t mode, const int32_t *block_table,
                                      int32_t table_stride, int32_t page_size, int32_t *out,
                                      void *stream) {
    return topk::launch_static(logits, row_stride, rows, width, valid_len, k, mode, block_table,
                               table_stride, page_size, out, stream);
}

topk_status_t topk_bf16_select_ex(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                  int32_t width, const int32_t *valid_len, int32_t k,
                                  topk_mode_t mode, const int32_t *block_table,
                                  int32_t table_stride, int32_t page_size, int32_t *out,
                                  void *stream, const topk_bf16_options_t *options) {
    return topk::launch(logits, row_stride, rows, width, valid_len, k, mode, block_table,
                        table_stride, page_size, page_size, 1, out, stream, options);
}

const char *topk_bf16_status_string(topk_status_t status) {
    switch (status) {
        case TOPK_OK: return "ok";
        case TOPK_ERR_ARG: return "invalid argument";
        case TOPK_ERR_ALIGN: return "misaligned logits, row stride, output or table";
        case TOPK_ERR_K: return "k outside [1, 2048]";
        case TOPK_ERR_WIDTH: return "width outside [0, 1048576] or row_stride < width";
        case TOPK_ERR_CUDA: return "CUDA error";
        case TOPK_ERR_SIZE: return "more rows or wider rows than topk_bf16_select_static takes";
    }
    return "unknown status";
}

topk_status_t topk_bf16_plan(int32_t rows, int32_t width, int32_t k, topk_mode_t mode,
                             int32_t *cluster, int32_t *threads, int32_t *smem_bytes,
                             int32_t *variant, int32_t *ctas) {
    if (rows < 0 || (mode != TOPK_TOKEN && mode != TOPK_BLOCK8)) return TOPK_ERR_ARG;
    if (k < 1 || k > TOPK_MAX_K) return TOPK_ERR_K;
    if (width < 0 || width > TOPK_MAX_WIDTH) return TOPK_ERR_WIDTH;
    int dev = 0;
    topk::DeviceInit *d = nullptr;
    if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (topk::init_device(dev, d) != cudaSuccess) return TOPK_ERR_CUDA;
    const bool block = mode == TOPK_BLOCK8;
    const topk::Plan pl = topk::make_plan(rows, width, k, *d, block, 0, 0);
    const topk::Variant v = pl.kind == topk::KIND_ONE ? topk::one_variant(block, pl.build)
                            : pl.kind == topk::KIND_STREAM ? topk::stream_variant(block) : topk::direct_variant(block);
    if (cluster) *cluster = pl.cluster;
    if (threads) *threads = pl.threads;
    if (smem_bytes) *smem_bytes = v.smem;
    if (variant) *variant = pl.kind;
    if (ctas) *ctas = static_cast<int32_t>(pl.clusters * pl.cluster);
    return TOPK_OK;
}

topk_status_t topk_bf16_device_status(uint32_t *flags, int32_t clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return TOPK_ERR_CUDA;
    uint32_t v = 0;
    for (auto f : {topk::status_stream, topk::status_direct, topk::status_one, topk::status_ordered}) {
        uint32_t u = 0;
        if (f(&u, clear != 0) != cudaSuccess) return TOPK_ERR_CUDA;
        v |= u;
    }
    if (flags) *flags = v;
    return TOPK_OK;
}

}  // extern "C"