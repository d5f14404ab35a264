// Launch parameters and the host-side interface between the library's
// translation units (plain C++: no device code).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace topk {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int VPT = 8;                       // 16-byte vectors per thread per tile
constexpr int TILE_VEC = THREADS * VPT;      // 2048 vectors = 32 KiB per stage
constexpr int QCAP = 32 * VPT;               // queue entries of one warp
constexpr int TIECAP = 256;                  // ties ranked directly
constexpr uint32_t KEY_POS_INF = 0xFF80u;    // key of +inf
constexpr uint32_t KEY_NEG_INF = 0x007Fu;    // key of -inf
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // a stage wait gives up after 1 s
constexpr uint32_t ALL = 0xFFFFFFFFu;        // "every tie" / "no cut"

enum : uint32_t { ERR_WAIT = 1u, ERR_BOUNDS = 2u, ERR_DEBUG_INDEX = 4u };

struct Params {
    const uint16_t *logits;
    int64_t row_stride;
    int32_t rows, width;
    const int32_t *valid_len;
    int32_t k;
    const int32_t *table;
    int32_t table_stride, page_shift;
    int32_t block_rows;                      // physical rows per page
    int32_t rows_per_request;                // rows sharing one table row
    int32_t *out;
    uint32_t *counters;
    int32_t force_direct;
    int32_t release;                         // 0: hold the next grid on the stream until this
                                             // one completes (see grid_dependents_release)
};

namespace ordered {
constexpr int NT = 512;
struct OParams {
    const uint16_t *logits;
    int64_t row_stride;
    int32_t rows, width;
    const int32_t *valid_len;
    int32_t k;
    const uint16_t *tops;        // NULL: every row takes the exact select
    int64_t tops_stride;
    const int32_t *table;
    int32_t table_stride, page_shift, block_rows, rows_per_request;
    int32_t *out, *valid, *ids;
    uint32_t *counters;
    int32_t words;        // 1: out holds B' words [rows, k + k / 32] (IndexerLocalTopk)
    int32_t release;      // as Params::release
};
}  // namespace ordered

namespace direct {
constexpr int NT = 256;
constexpr int RES = 16384;                   // resident keys per CTA
}  // namespace direct

// A kernel and the dynamic shared memory it is launched with.
struct Variant {
    const void *fn;
    int smem;
};

// Defined by the kernels' translation units.
Variant stream_variant(bool block);               // stream.cu: the streamed cluster kernel
Variant direct_variant(bool block);               // direct.cu: the resident-keys kernel
constexpr int ONE_BUILDS = 3;                     // one-tile builds (see one_variant)
constexpr int one_threads(int build) { return build == 2 ? 512 : 256; }
Variant one_variant(bool block, int build);       // one_tile.cu: the one-tile kernel
Variant one_static_variant(bool block, int build);  // one_tile.cu: topk_bf16_select_static's kernel
cudaError_t static_row_carry(int dev, uint32_t **table);  // one_tile.cu: its table, set up once per device
Variant ordered_variant();                        // ordered.cu: the ordered kernel
cudaError_t launch_tops(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                        const int32_t *valid_len, uint16_t *tops, int64_t tops_stride, int32_t pieces,
                        unsigned blocks, cudaStream_t stream);
// The device status word of each translation unit: read (and zero when clear).
cudaError_t status_stream(uint32_t *v, bool clear);
cudaError_t status_direct(uint32_t *v, bool clear);
cudaError_t status_one(uint32_t *v, bool clear);
cudaError_t status_ordered(uint32_t *v, bool clear);

}  // namespace topk
