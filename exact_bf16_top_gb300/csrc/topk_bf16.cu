// Exact per-row top-k of BF16 logits for GB300 (sm_103a).
//
// The operation: vLLM "decode_topk_cute", module docstring ("What this module
// computes"); the order key and NaN rule: sglang PR #39305 "Exact bf16 consumer
// top-k adapted from DeepSelect", Modifications; lowest-index ties and the
// block-table transform: vLLM kimi_k3 "dsa/indexer", IndexerSelect.
//
// Design. A row is split over a cluster of C CTAs (C in {1, 2, 4, 8, 16}); each
// CTA owns a contiguous share of the row's valid 16-byte vectors. Clusters are
// persistent: each one walks its rows in turn, and one thread keeps a ring of
// 32 KiB shared-memory stages filled with bulk async copies (cp.async.bulk +
// mbarrier) that runs ahead across row boundaries, so the next row streams in
// while the current one is being selected.
//
// Every CTA keeps a candidate buffer of (key, index) pairs in shared memory, in
// no particular order: it always holds every key of the CTA's share that can
// still be selected, plus some that cannot. Ties at a cutoff are settled by
// index only when they have to be (the lowest indices win): usually a handful
// of entries ranked directly, a two-pass radix select over the indices when
// there are many.
//
// The first stage ("tile": 256 threads x 8 vectors) of a CTA's share is
// selected exactly. Its cutoff comes from group representatives: each thread
// splits its logits into groups of g and takes one element of each group, the
// packed signed maximum of its BF16 bits (the group maximum whenever the group
// holds a non-negative value). The k-th largest representative, found with a
// 12-bit histogram, bounds the tile's k-th key from below, because k distinct
// elements reach it; keys above it sit in about k groups, so they are few. Those
// survivors go to the buffer and their exact k-th comes from a histogram
// relative to the cutoff. When the representatives cannot bound the tile, or
// the survivors overflow, every key becomes its own representative (g = 1): the
// exact path. Later tiles append every key at or above a running threshold,
// which rises whenever the buffer is compacted to its top-k and, in a cluster,
// when a peer CTA publishes its own bound through distributed shared memory.
//
// A vector is first tested on its packed maximum; the vectors that may hold a
// wanted key are queued per warp (ballots), and the warp's lanes work through
// the queue together, so divergence does not multiply the work; a warp
// reserves its slots with one shared atomic, never one per key. The C buffers
// of a row are merged with cluster-wide histograms over distributed shared
// memory; ties at the row's k-th key are split across CTAs in index order, and
// each CTA writes its part of the answer through the block table.
// All selection arithmetic is on 16-bit integer keys; no floating point.

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "topk_bf16.h"

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

enum : uint32_t { ERR_WAIT = 1u, ERR_BOUNDS = 2u };

__device__ uint32_t g_device_status;

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

template <int NSTAGE, int CAP>
struct alignas(128) Smem {
    uint4 stage[NSTAGE][TILE_VEC];           // streamed logits
    uint32_t buf_idx[CAP];                   // candidate buffer (any order)
    uint16_t buf_key[CAP];
    alignas(16) uint32_t hwin[4][256];       // window histograms (zero between uses); [1]: the
                                             // running histogram of the buffer (see filter_tile)
    uint32_t h_merge[2][256];                // this CTA's merge histograms (peers read them)
    uint32_t m_all[256];                     // merge: counts over the cluster
    uint32_t m_pre[2][256];                  // merge: counts over lower-ranked CTAs
    uint32_t tie_idx[TIECAP];                // indices of ties being ranked
    uint32_t red[2][WARPS];                  // block-scan warp totals
    uint32_t bc[4];                          // broadcast words
    uint32_t v_count;                        // buffer entries
    uint32_t v_bufmax;                       // largest buffer key (buffer_max's scratch)
    uint32_t v_ntie, v_emit, v_flag;
    uint32_t v_full[2];                      // a warp found the buffer full, by tile parity
    uint32_t v_arrive[2];                    // warps done appending, by tile parity
    uint32_t v_newthr;                       // a raised threshold for the next tile (0: none)
    uint32_t shared_thr[2];                  // lower bound on the row's k-th key (max), by row parity
    uint32_t shared_max[2];                  // largest candidate key of the row (max), by row parity
    uint32_t thr_snap;                       // shared_thr as every thread sees it this tile
    uint32_t abort_flag;                     // a bounded wait gave up
    uint16_t queue[WARPS][QCAP];             // per-warp vector queues (tile positions)
    unsigned long long full[NSTAGE];         // stage mbarriers
};

// --------------------------------------------------------------------- PTX bits

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Bulk async copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for a stage: gives up after WAIT_LIMIT_NS (recording ERR_WAIT and
// raising the CTA's abort flag, which ends every later wait at once).
__device__ __forceinline__ void mbar_wait(unsigned long long *bar, uint32_t parity,
                                          volatile uint32_t *abort) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return;
        if (*abort) return;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
            *abort = 1u;
            atomicOr(&g_device_status, ERR_WAIT);
            return;
        }
    }
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t peer_addr(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_peer(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Word w of every CTA of the cluster: the sum over all of them and over those
// ranked below this one. The C loads are issued back to back (one round trip).
__device__ __forceinline__ void cluster_sum(const uint32_t *w, uint32_t C, uint32_t rank, uint32_t &all,
                                            uint32_t &pre) {
    uint32_t x[16];
#pragma unroll
    for (uint32_t r = 0; r < 16; ++r) x[r] = r < C ? ld_peer(peer_addr(w, r)) : 0u;
    all = pre = 0u;
#pragma unroll
    for (uint32_t r = 0; r < 16; ++r) {
        all += x[r];
        pre += r < rank ? x[r] : 0u;
    }
}

__device__ __forceinline__ void red_max_peer(uint32_t addr, uint32_t v) {
    asm volatile("red.relaxed.cluster.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(v)
                 : "memory");
}

// Programmatic dependent launch (the DecodeTopK page's synchronisation notes:
// wait for the preceding grid before reading inputs, let the next one start
// early): the wait returns once the preceding grid has completed and its writes
// are visible; the release lets the next grid's CTAs start their prologue on
// free SMs while this one runs (they wait the same way before reading). A
// launch with the hold option skips the release, for a next kernel that reads
// this one's output without waiting first (IndexerSelect's release flag on the
// indexer page): that kernel then starts only once this grid has completed.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dependents_release() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Packed 16-bit maxima (signed / unsigned).
__device__ __forceinline__ uint32_t smax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.s16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t umax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// The larger half of a packed pair, as a signed / unsigned 16-bit value.
__device__ __forceinline__ int32_t smax_halves(uint32_t m) {
    return static_cast<int16_t>(smax2(m, __byte_perm(m, 0, 0x1032)) & 0xFFFFu);
}

__device__ __forceinline__ uint32_t umax_halves(uint32_t m) {
    return umax2(m, __byte_perm(m, 0, 0x1032)) & 0xFFFFu;
}

__device__ __forceinline__ uint32_t vec_smax(const uint4 &r) {
    return smax2(smax2(r.x, r.y), smax2(r.z, r.w));
}

// --------------------------------------------------------------------- keys

// Order-preserving keys of two packed BF16 values: x ^ (x < 0 ? 0xFFFF : 0x8000)
// per half (sglang PR #39305, Modifications).
__device__ __forceinline__ uint32_t key2(uint32_t w) {
    const uint32_t s = w & 0x80008000u;
    return w ^ (s - (s >> 15)) ^ 0x80008000u;
}

// Nonzero when either half is a NaN (exponent all ones, mantissa nonzero).
__device__ __forceinline__ uint32_t nan2(uint32_t w) {
    return ((w & 0x7FFF7FFFu) + 0x007F007Fu) & 0x80008000u;
}

// The key of the element whose BF16 bits, read as a signed 16-bit integer, are
// r (the result of a packed signed maximum), or 0 when it may not be used as a
// representative: NaN, below thr, or the pattern 0x8000 that marks lanes with
// no element.
__device__ __forceinline__ uint32_t rep_key(int32_t r, uint32_t thr) {
    const uint32_t bits = static_cast<uint32_t>(r) & 0xFFFFu;
    const uint32_t key = r >= 0 ? bits + 0x8000u : bits ^ 0xFFFFu;
    return (r != -32768 && key >= thr && key >= KEY_NEG_INF && key <= KEY_POS_INF) ? key : 0u;
}

// Token mode: an element is one logit. clean(): the keys of a vector's eight
// logits where eligible (not NaN, inside the valid length), else 0.
struct TokenMode {
    static constexpr bool BLOCK = false;
    static constexpr int KPV = 8;
    static constexpr int GMAX = 64;
    static constexpr uint32_t KMIN = KEY_NEG_INF;
    __device__ static __forceinline__ int32_t elem(int64_t v, int h) {
        return static_cast<int32_t>(v * 8 + h);
    }
    __device__ static __forceinline__ void clean(const uint4 &raw, int64_t v, int64_t V, int32_t L,
                                                 uint32_t (&ck)[4]) {
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        const int lanes = (v == V - 1) ? static_cast<int>(L - 8 * v) : 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t k = key2(w[i]);
            uint32_t lo = k & 0xFFFFu, hi = k >> 16;
            lo = (2 * i < lanes && lo >= KMIN && lo <= KEY_POS_INF) ? lo : 0u;
            hi = (2 * i + 1 < lanes && hi >= KMIN && hi <= KEY_POS_INF) ? hi : 0u;
            ck[i] = lo | (hi << 16);
        }
    }
    // Could the vector hold a key >= lim? (A superset test.)
    __device__ static __forceinline__ bool may_reach(const uint4 &raw, uint32_t ek, uint32_t lim) {
        (void)ek;
        if (lim > KEY_POS_INF) return false;
        if (lim >= 0x8000u) {
            // Keys >= 0x8000 are the non-negative values, whose keys are their
            // bits + 0x8000: compare the raw bits as signed 16-bit integers.
            return smax_halves(vec_smax(raw)) >= static_cast<int32_t>(lim - 0x8000u);
        }
        if (lim <= KMIN) return true;
        return umax_halves(umax2(umax2(key2(raw.x), key2(raw.y)), umax2(key2(raw.z), key2(raw.w)))) >= lim;
    }
};

// Block mode: an element is a vector, its key the NaN-propagating maximum of
// its eight logits; the newest block is pinned at +inf; NaN blocks and -inf
// blocks are ineligible (a selected -inf block is written as -1, which is what
// an unfilled slot holds anyway).
struct BlockMode {
    static constexpr bool BLOCK = true;
    static constexpr int KPV = 1;
    static constexpr int GMAX = 4;
    static constexpr uint32_t KMIN = KEY_NEG_INF + 1;
    __device__ static __forceinline__ int32_t elem(int64_t v, int) { return static_cast<int32_t>(v); }
    __device__ static __forceinline__ uint32_t key(const uint4 &raw, int64_t v, int64_t V) {
        if (v == V - 1) return KEY_POS_INF;
        if (nan2(raw.x) | nan2(raw.y) | nan2(raw.z) | nan2(raw.w)) return 0u;
        const uint32_t k =
            umax_halves(umax2(umax2(key2(raw.x), key2(raw.y)), umax2(key2(raw.z), key2(raw.w))));
        return k >= KMIN ? k : 0u;
    }
    __device__ static __forceinline__ void clean(const uint4 &raw, int64_t v, int64_t V, int32_t,
                                                 uint32_t (&ck)[4]) {
        ck[0] = key(raw, v, V);
        ck[1] = ck[2] = ck[3] = 0u;
    }
    __device__ static __forceinline__ bool may_reach(const uint4 &, uint32_t ek, uint32_t lim) {
        return ek >= lim && ek != 0u;
    }
};

template <class M>
__device__ __forceinline__ uint32_t key_at(const uint32_t (&ck)[4], int h) {
    return M::BLOCK ? ck[0] : (ck[h >> 1] >> ((h & 1) * 16)) & 0xFFFFu;
}

// ------------------------------------------------------------- warp primitives

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// Exclusive prefix over the warp of counts in [0, 15], and their total: four
// ballots of the count's bits instead of a shuffle scan.
__device__ __forceinline__ uint32_t warp_excl_small(uint32_t cnt, uint32_t &total) {
    const uint32_t lt = (1u << lane_id()) - 1u;
    const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, cnt & 1u), b1 = __ballot_sync(0xFFFFFFFFu, cnt & 2u);
    const uint32_t b2 = __ballot_sync(0xFFFFFFFFu, cnt & 4u), b3 = __ballot_sync(0xFFFFFFFFu, cnt & 8u);
    total = __popc(b0) + 2u * __popc(b1) + 4u * __popc(b2) + 8u * __popc(b3);
    return __popc(b0 & lt) + 2u * __popc(b1 & lt) + 4u * __popc(b2 & lt) + 8u * __popc(b3 & lt);
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
    const uint32_t lane = lane_id();
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, d);
        if (lane >= static_cast<uint32_t>(d)) v += t;
    }
    return v;
}

// The bin b of a 256-bin histogram that holds the q-th largest key: above =
// count in bins > b, above < q <= above + count(b). Run by a whole warp; every
// warp that runs it gets the same answer. Returns false if the total is < q.
__device__ __forceinline__ bool find_bin256(const uint32_t *hist, uint32_t q, uint32_t &bin,
                                            uint32_t &above, uint32_t &total) {
    // A warp that reaches this diverged (after leader-only atomics, say) would
    // run the scan below split in lane groups: reconverge first.
    __syncwarp();
    const uint32_t lane = lane_id();
    const int lo_bin = 248 - 8 * static_cast<int>(lane);
    const uint4 a = *reinterpret_cast<const uint4 *>(hist + lo_bin);
    const uint4 b = *reinterpret_cast<const uint4 *>(hist + lo_bin + 4);
    const uint32_t h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += h[i];
    const uint32_t incl = warp_incl_scan(s);
    total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl >= q);
    if (hit == 0) {
        bin = 0;
        above = total;
        return false;
    }
    const int src = __ffs(hit) - 1;
    uint32_t my_bin = 0, my_above = 0;
    if (static_cast<int>(lane) == src) {
        uint32_t acc = incl - s;
        bool done = false;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
            if (!done && acc + h[i] >= q) {
                my_bin = static_cast<uint32_t>(lo_bin + i);
                my_above = acc;
                done = true;
            }
            acc += h[i];
        }
    }
    bin = __shfl_sync(0xFFFFFFFFu, my_bin, src);
    above = __shfl_sync(0xFFFFFFFFu, my_above, src);
    return true;
}

__device__ __forceinline__ void count_event(const Params &p, int which) {
    if (p.counters && threadIdx.x == 0) atomicAdd(p.counters + which, 1u);
}

// Cycle accounting for the diagnosis counters (thread 0, only when enabled).
struct PhaseClock {
    long long t = 0;
    __device__ __forceinline__ void start(const Params &p) {
        if (p.counters && threadIdx.x == 0) t = clock64();
    }
    __device__ __forceinline__ void stop(const Params &p, int which) {
        if (p.counters && threadIdx.x == 0)
            atomicAdd(p.counters + which, static_cast<uint32_t>(clock64() - t));
    }
};

// The table row of a row: its request's (IndexerSelect: request = row / q).
__device__ __forceinline__ const int32_t *table_row(const Params &p, int32_t row) {
    const int32_t request = p.rows_per_request == 1 ? row : row / p.rows_per_request;
    return p.table + static_cast<int64_t>(request) * p.table_stride;
}

// Page of element i times the physical rows per page, plus i's offset in its
// page (IndexerSelect.emit).
__device__ __forceinline__ int32_t transform(const Params &p, int32_t row, int32_t i) {
    if (!p.table) return i;
    const int32_t page = table_row(p, row)[i >> p.page_shift];
    return page * p.block_rows + (i & ((1 << p.page_shift) - 1));
}

// Warp-aggregated reservation of `n` slots (lane 0 adds; every lane gets base).
__device__ __forceinline__ uint32_t warp_reserve(uint32_t *ctr, uint32_t n) {
    uint32_t base = 0;
    if (lane_id() == 0 && n) base = atomicAdd(ctr, n);
    return __shfl_sync(0xFFFFFFFFu, base, 0);
}

// --------------------------------------------------------- the CTA's machinery
//
// The per-row state is uniform across the CTA and lives in registers; every
// routine is inlined so that the compiler sees shared-memory accesses as such
// (out of line, they would go through generic addresses).

// Add 1 for every lane with `valid`, one shared atomic per distinct bin in the
// warp (a crowded bin would otherwise serialise the atomics of the whole warp).
__device__ __forceinline__ void agg_add(uint32_t *hist, uint32_t bin, bool valid) {
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, valid ? bin : 0xFFFFFFFFu);
    if (valid && lane_id() == static_cast<uint32_t>(__ffs(peers) - 1)) atomicAdd(&hist[bin], __popc(peers));
    __syncwarp();  // reconverge after the leaders' atomics
}

template <class M, int NSTAGE, int CAP>
struct Cta {
    static constexpr int KPV = M::KPV;
    using S = Smem<NSTAGE, CAP>;

    S *s;
    const Params *p;
    uint32_t C = 1, rank = 0;
    uint32_t parity = 0;     // alternates double-buffered scan scratch
    uint32_t slot = 0;       // parity of this cluster's row: which shared words it uses
    int32_t row = 0, L = 0;
    int64_t V = 0;
    uint32_t k = 0;
    uint32_t thr = 0;        // keep keys >= thr
    uint32_t buf_lo = 0;     // every buffer key is >= buf_lo
    uint32_t best_T = 0;     // largest lower bound on the row's k-th key found here
    uint32_t tpar = 0;       // parity of the filter tiles: picks s->v_full, s->v_arrive
    uint32_t f_Q = 0, f_next = 0, f_lim = 0;  // this warp's queue, where its appends stopped, the limit
    uint32_t first_c = 0;    // the first tile's cut while its ties are pending (0: none)
    bool f_fast = false;
    bool run_ok = false;     // s->hwin[1] counts every buffer key >= run_lo, in bins key - run_lo
    uint32_t run_lo = 0;     // (the top bin also holding every key >= run_lo + 255)

    __device__ __forceinline__ static uint32_t volatile_load(const uint32_t *x) {
        return *reinterpret_cast<const volatile uint32_t *>(x);
    }

    // The threshold with the peers' bound as of the last snapshot (the same in
    // every thread: thread 0 takes the snapshot before a barrier).
    __device__ __forceinline__ uint32_t effective_thr() const { return C > 1 ? max(thr, s->thr_snap) : thr; }

    __device__ __forceinline__ void snapshot_shared() {
        if (C > 1 && threadIdx.x == 0) s->thr_snap = volatile_load(&s->shared_thr[slot]);
    }

    // Every CTA of the row learns that the row's k-th key is at least `bound`.
    __device__ __forceinline__ void publish(uint32_t bound) {
        best_T = max(best_T, bound);
        if (C > 1 && threadIdx.x < C && threadIdx.x != rank)
            red_max_peer(peer_addr(&s->shared_thr[slot], threadIdx.x), bound);
    }

    __device__ __forceinline__ void clean_at(const uint4 *stg, int64_t tile_v0, int pos, uint32_t (&ck)[4]) const {
        M::clean(stg[pos], tile_v0 + pos, V, L, ck);
    }

    // Inclusive scan over the CTA's threads (one __syncthreads).
    __device__ __forceinline__ uint32_t block_incl_scan(uint32_t x, uint32_t &total) {
        const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
        const uint32_t inc = warp_incl_scan(x);
        if (lane == 31) s->red[parity][warp] = inc;
        __syncthreads();
        const uint32_t w = lane < WARPS ? s->red[parity][lane] : 0u;
        const uint32_t wi = warp_incl_scan(w);
        total = __shfl_sync(0xFFFFFFFFu, wi, 31);
        const uint32_t pre = __shfl_sync(0xFFFFFFFFu, wi - w, warp);
        parity ^= 1u;
        return pre + inc;
    }

    // Bin of `key` in a window [lo, lo + (256 << shift)); a key outside it would
    // break the caller's bounds, so it is recorded and clamped.
    __device__ __forceinline__ static uint32_t window_bin(uint32_t key, uint32_t lo, int shift) {
        const uint32_t o = (key - lo) >> shift;
        if (key < lo || o > 255u) {
            atomicOr(&g_device_status, ERR_BOUNDS);
            return key < lo ? 0u : 255u;
        }
        return o;
    }

    // The q-th largest of buf_key[first .. first + n), all within [lo, hi]
    // (q <= n): radix select over bins relative to lo, one pass when hi - lo <
    // 256, else two. T = that key, above = keys greater than it. Uses
    // s->hwin[2] and s->hwin[3] (zero on entry and on exit).
    __device__ __forceinline__ void window_select(uint32_t first, uint32_t n, uint32_t lo, uint32_t hi,
                                               uint32_t q, uint32_t *T_out, uint32_t *above_out) {
        const int tid = threadIdx.x;
        const uint32_t range = hi - lo;
        const int shift = range < 256u ? 0 : (32 - __clz(static_cast<int>(range))) - 8;
        for (uint32_t i = tid; i < n; i += THREADS) {
            const uint32_t key = s->buf_key[first + i];
            if (key != 0u) atomicAdd(&s->hwin[2][window_bin(key, lo, shift)], 1u);  // 0: a dead entry
        }
        __syncthreads();
        uint32_t b1, above1, tot, T, above;
        find_bin256(s->hwin[2], q, b1, above1, tot);
        if (shift == 0) {
            T = lo + b1;
            above = above1;
        } else {
            const uint32_t mask = (1u << shift) - 1u;
            for (uint32_t i = tid; i < n; i += THREADS) {
                const uint32_t key = s->buf_key[first + i];
                const uint32_t o = key - lo;
                if (key != 0u && (o >> shift) == b1) atomicAdd(&s->hwin[3][o & mask], 1u);
            }
            __syncthreads();
            uint32_t b2, above2;
            find_bin256(s->hwin[3], q - above1, b2, above2, tot);
            T = lo + (b1 << shift) + b2;
            above = above1 + above2;
        }
        __syncthreads();
        s->hwin[2][tid] = 0u;
        s->hwin[3][tid] = 0u;
        *T_out = T;
        *above_out = above;
    }

    // The q-th smallest index among buffer entries [0, n) whose key is T, when
    // there are more than TIECAP of them: a two-pass radix select over 10-bit
    // digits (indices are below 2^20), in the 1024 words of s->hwin (zero on
    // entry and on exit).
    __device__ __forceinline__ uint32_t tie_radix(uint32_t n, uint32_t T, uint32_t q) {
        const int tid = threadIdx.x;
        uint32_t cut = 0, need = q;
        for (int pass = 0; pass < 2; ++pass) {
            const int sh = pass == 0 ? 10 : 0;
            for (uint32_t i = tid; i < n; i += THREADS) {
                if (s->buf_key[i] != T) continue;
                const uint32_t x = s->buf_idx[i];
                if (pass == 1 && (x >> 10) != (cut >> 10)) continue;
                atomicAdd(&s->hwin[0][(x >> sh) & 1023u], 1u);
            }
            __syncthreads();
            uint4 *h4 = reinterpret_cast<uint4 *>(&s->hwin[0][0]) + tid;  // bins [4t, 4t + 4), ascending
            const uint4 hv = *h4;
            *h4 = make_uint4(0, 0, 0, 0);
            const uint32_t v[4] = {hv.x, hv.y, hv.z, hv.w};
            const uint32_t sum = v[0] + v[1] + v[2] + v[3];
            uint32_t total;
            const uint32_t incl = block_incl_scan(sum, total);
            uint32_t acc = incl - sum;
            if (acc < need && need <= incl) {
                bool done = false;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (!done && acc + v[i] >= need) {
                        s->bc[0] = static_cast<uint32_t>(4 * tid + i);
                        s->bc[1] = acc;
                        done = true;
                    }
                    acc += v[i];
                }
            }
            __syncthreads();
            cut |= s->bc[0] << sh;
            need -= s->bc[1];
        }
        return cut;
    }

    // Among buffer entries [0, n) with key T (distinct indices), the cut with
    // exactly q of them at or below it; ALL when q covers them all.
    __device__ __forceinline__ uint32_t tie_cut(uint32_t n, uint32_t T, uint32_t q) {
        const int tid = threadIdx.x;
        const uint32_t lt = (1u << lane_id()) - 1u;
        __syncthreads();
        if (tid == 0) s->v_ntie = 0u;
        __syncthreads();
        for (uint32_t i0 = 0; i0 < n; i0 += THREADS) {
            const uint32_t i = i0 + tid;
            const bool tie = i < n && s->buf_key[i] == T;
            const uint32_t b = __ballot_sync(0xFFFFFFFFu, tie);
            const uint32_t at = warp_reserve(&s->v_ntie, __popc(b)) + __popc(b & lt);
            if (tie && at < static_cast<uint32_t>(TIECAP)) s->tie_idx[at] = s->buf_idx[i];
        }
        __syncthreads();
        const uint32_t e = s->v_ntie;
        if (q >= e) return ALL;
        if (e > static_cast<uint32_t>(TIECAP)) return tie_radix(n, T, q);
        if (static_cast<uint32_t>(tid) < e) {
            const uint32_t mine = s->tie_idx[tid];
            uint32_t r = 0;
            for (uint32_t u = 0; u < e; ++u) r += s->tie_idx[u] < mine;
            if (r == q - 1) s->bc[3] = mine;
        }
        __syncthreads();
        return s->bc[3];
    }

    // Queue, per warp and in index order, the tile's vectors that may hold a
    // key >= lim. Returns the queue length.
    __device__ __forceinline__ uint32_t build_queue(const uint4 *stg, int64_t tile_v0, int nv, uint32_t lim) {
        const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
        const uint32_t lt = (1u << lane) - 1u;
        uint32_t q = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int pos = j * THREADS + static_cast<int>(threadIdx.x);
            bool pass = false;
            if (pos < nv) {
                const uint4 raw = stg[pos];
                pass = M::may_reach(raw, M::BLOCK ? BlockMode::key(raw, tile_v0 + pos, V) : 0u, lim);
            }
            const uint32_t b = __ballot_sync(0xFFFFFFFFu, pass);
            if (pass) s->queue[warp][q + __popc(b & lt)] = static_cast<uint16_t>(j * THREADS + static_cast<int>(threadIdx.x));
            q += __popc(b);
        }
        __syncwarp();
        return q;
    }

    __device__ __forceinline__ int queued_pos(uint32_t e) const {
        return static_cast<int>(s->queue[threadIdx.x >> 5][e]);
    }

    // Append every key >= lim of this warp's queued vectors, from queue entry
    // `from` on, to the buffer (any order). Slots are reserved a warp at a time
    // and only while they fit. Returns the first entry not appended (Q: all).
    __device__ __forceinline__ uint32_t append_keys(const uint4 *stg, int64_t tile_v0, uint32_t Q,
                                                 uint32_t from, uint32_t lim) {
        const uint32_t lane = lane_id();
        for (uint32_t e0 = from; e0 < Q; e0 += 32) {
            const uint32_t e = e0 + lane;
            uint32_t ck[4] = {0u, 0u, 0u, 0u};
            int pos = 0;
            if (e < Q) {
                pos = queued_pos(e);
                clean_at(stg, tile_v0, pos, ck);
            }
            uint32_t cnt = 0;
#pragma unroll
            for (int h = 0; h < KPV; ++h) {
                const uint32_t key = key_at<M>(ck, h);
                cnt += key >= lim;
            }
            uint32_t total, at;
            const uint32_t before = warp_excl_small(cnt, total);
            if (!reserve(total, before, cnt, at)) return e0;  // full: the caller compacts and resumes here
            if (cnt) {
#pragma unroll
                for (int h = 0; h < KPV; ++h) {
                    const uint32_t key = key_at<M>(ck, h);
                    if (key >= lim) {
                        s->buf_key[at] = static_cast<uint16_t>(key);
                        s->buf_idx[at] = M::elem(tile_v0 + pos, h);
                        if (run_ok) atomicAdd(&s->hwin[1][min(key - run_lo, 255u)], 1u);
                        ++at;
                    }
                }
            }
        }
        return Q;
    }

    // Slots for a warp's `total` new entries (lane 0 adds; every lane learns
    // the base); `at` = this lane's first slot, `before` entries of lower lanes
    // precede it. When the buffer cannot hold them all, the warp's slots below
    // CAP get key 0 (an entry nothing counts or selects) and false is returned:
    // the caller compacts and resumes. Reservations only grow, so every later
    // one fails too.
    __device__ __forceinline__ bool reserve(uint32_t total, uint32_t before, uint32_t cnt, uint32_t &at) {
        uint32_t base = 0;
        if (lane_id() == 0 && total) base = atomicAdd(&s->v_count, total);
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
        at = base + before;
        if (base + total <= static_cast<uint32_t>(CAP)) return true;
        for (uint32_t i = at; i < at + cnt && i < static_cast<uint32_t>(CAP); ++i) s->buf_key[i] = 0u;
        return false;
    }

    // publish() from any one warp: lane r tells peer r.
    __device__ __forceinline__ void publish_lane(uint32_t bound) {
        const uint32_t lane = lane_id();
        best_T = max(best_T, bound);
        if (C > 1 && lane < C && lane != rank) red_max_peer(peer_addr(&s->shared_thr[slot], lane), bound);
    }

    // Token mode, lim >= 0x8000: the keys >= lim are the non-negative values
    // whose BF16 bits, as signed 16-bit integers, are >= lim - 0x8000 (NaN is
    // excluded by setting its sign bit first). These are build_queue and
    // append_keys for that case, on raw bits: no key conversion per element.
    __device__ __forceinline__ uint32_t build_queue_fast(const uint4 *stg, int nv, int32_t cs) {
        const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
        const uint32_t lt = (1u << lane) - 1u;
        uint32_t q = 0;
        int32_t mx[VPT];  // every vector's maximum first: the loads issue together
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int pos = j * THREADS + static_cast<int>(threadIdx.x);
            mx[j] = pos < nv ? smax_halves(vec_smax(stg[pos])) : -32768;
        }
        uint32_t b[VPT];  // every ballot first: the stores then only wait on popcounts
#pragma unroll
        for (int j = 0; j < VPT; ++j) b[j] = __ballot_sync(0xFFFFFFFFu, mx[j] >= cs);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (mx[j] >= cs) s->queue[warp][q + __popc(b[j] & lt)] = static_cast<uint16_t>(j * THREADS + static_cast<int>(threadIdx.x));
            q += __popc(b[j]);
        }
        __syncwarp();
        return q;
    }

    __device__ __forceinline__ uint32_t append_fast(const uint4 *stg, int64_t tile_v0, uint32_t Q,
                                                 uint32_t from, uint32_t lim) {
        const uint32_t lane = lane_id();
        const int32_t cs = static_cast<int32_t>(lim) - 0x8000;
        const uint32_t csm = (static_cast<uint32_t>(cs - 1) & 0xFFFFu) * 0x10001u;
        for (uint32_t e0 = from; e0 < Q; e0 += 32) {
            const uint32_t e = e0 + lane;
            uint32_t m = 0;
            int pos = 0;
            uint4 r = make_uint4(0, 0, 0, 0);
            if (e < Q) {
                pos = queued_pos(e);
                r = stg[pos];
                const uint32_t w[4] = {r.x, r.y, r.z, r.w};
                uint32_t u = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t x = w[i] | nan2(w[i]);
                    const uint32_t g = smax2(x, csm) ^ csm;  // nonzero halves: x >= cs
                    u |= ((((g & 0x7FFF7FFFu) + 0x7FFF7FFFu) | g) & 0x80008000u) >> (15 - i);
                }
                m = (u & 0xFu) | ((u >> 12) & 0xF0u);  // bit i: low half of word i; bit 4 + i: high half
            }
            const uint32_t cnt = __popc(m);
            uint32_t total, at;
            const uint32_t before = warp_excl_small(cnt, total);
            if (!reserve(total, before, cnt, at)) return e0;  // full: the caller compacts and resumes here

            const uint32_t idx0 = static_cast<uint32_t>(tile_v0 + pos) * 8u;
#pragma unroll 1
            for (; m; m &= m - 1u) {
                const int bit = __ffs(m) - 1;
                const int i = bit & 3, hi = bit >> 2;
                const uint32_t w = i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w;
                const uint32_t key = ((hi ? w >> 16 : w) & 0xFFFFu) + 0x8000u;
                s->buf_key[at] = static_cast<uint16_t>(key);
                s->buf_idx[at] = idx0 + static_cast<uint32_t>(2 * i + hi);
                if (run_ok) atomicAdd(&s->hwin[1][min(key - run_lo, 255u)], 1u);
                ++at;
            }
        }
        return Q;
    }

    // Token mode: the row's last vector, when partial, gets 0x8000 (a negative
    // value no cut selects) in the lanes past the valid length, by the thread
    // that owns its position in this tile (its warp reads it after a warp
    // barrier).
    __device__ __forceinline__ void mask_tail(const uint4 *stg, int64_t tile_v0, int nv) const {
        if (M::BLOCK || (L & 7) == 0) return;
        const int64_t pos = V - 1 - tile_v0;
        if (pos < 0 || pos >= nv || static_cast<int>(pos % THREADS) != static_cast<int>(threadIdx.x)) return;
        uint4 *v = const_cast<uint4 *>(stg) + pos;
        const int lanes = L & 7;
        const uint4 r = *v;
        uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int h = 0; h < 8; ++h)
            if (h >= lanes)
                w[h >> 1] = (w[h >> 1] & ((h & 1) ? 0x0000FFFFu : 0xFFFF0000u)) |
                            ((h & 1) ? 0x80000000u : 0x00008000u);
        *v = make_uint4(w[0], w[1], w[2], w[3]);
    }

    // Feed the tile's group representatives, as keys, to the high-byte
    // histogram s->hwin[2] (hb == ALL), or those whose high byte is hb to the
    // low-byte histogram s->hwin[3]. A representative is one element of a group
    // of g logits (token) or g blocks (block), with key >= thr, or nothing;
    // g = 1 feeds every candidate key. Every lane of a warp feeds together.
    __device__ __forceinline__ void rep_pass(const uint4 *stg, int64_t tile_v0, int nv, uint32_t g, uint32_t hb) {
        rep_walk(stg, tile_v0, nv, g, [&](uint32_t key) {
            if (hb == ALL) agg_add(s->hwin[2], key >> 8, key != 0u);
            else agg_add(s->hwin[3], key & 0xFFu, key != 0u && (key >> 8) == hb);
        });
    }

    // The tile's representatives (groups of g, keys >= thr, else 0) fed to
    // feed(key), every lane of a warp together.
    template <class F>
    __device__ __forceinline__ void rep_walk(const uint4 *stg, int64_t tile_v0, int nv, uint32_t g, F &&feed) {
        uint32_t acc = 0x80008000u;   // token: packed running maximum of a group
        uint32_t bacc = 0u;           // block: running maximum key of a group
        const uint32_t per = g >= 8u ? g >> 3 : 1u;  // vectors per token group
        for (int j = 0; j < VPT; ++j) {
            const int pos = j * THREADS + static_cast<int>(threadIdx.x);
            const int64_t v = tile_v0 + pos;
            if constexpr (M::BLOCK) {
                const uint32_t key = pos < nv ? BlockMode::key(stg[pos], v, V) : 0u;
                bacc = max(bacc, key);
                if (((j + 1) & (g - 1u)) == 0u) {
                    feed(bacc >= thr ? bacc : 0u);
                    bacc = 0u;
                }
            } else {
                const bool usable = pos < nv && !(v == V - 1 && (L & 7));
                if (g == 1u) {
                    uint32_t ck[4] = {0u, 0u, 0u, 0u};
                    if (pos < nv) clean_at(stg, tile_v0, pos, ck);
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const uint32_t key = key_at<M>(ck, h);
                        feed(key >= thr ? key : 0u);
                    }
                } else if (g == 4u) {
                    const uint4 r = usable ? stg[pos] : make_uint4(0x80008000u, 0x80008000u, 0x80008000u, 0x80008000u);
                    feed(rep_key(smax_halves(smax2(r.x, r.y)), thr));
                    feed(rep_key(smax_halves(smax2(r.z, r.w)), thr));
                } else {
                    if (usable) acc = smax2(acc, vec_smax(stg[pos]));
                    if ((static_cast<uint32_t>(j) + 1u) % per == 0u) {
                        feed(rep_key(smax_halves(acc), thr));
                        acc = 0x80008000u;
                    }
                }
            }
        }
    }

    // The `take` lowest-index keys equal to c in the tile, appended at
    // first .. first + take, found with ordered scans of per-vector tie counts
    // (tile order is index order: vector j * THREADS + thread, then lane). For
    // tiles whose cut sits in a crowded bin.
    __device__ __forceinline__ void ordered_ties(const uint4 *stg, int64_t tile_v0, int nv, uint32_t c,
                                              uint32_t take, uint32_t first) {
        uint32_t before = 0;
        for (int j = 0; j < VPT && before < take; ++j) {
            const int pos = j * THREADS + static_cast<int>(threadIdx.x);
            uint32_t ck[4] = {0u, 0u, 0u, 0u};
            if (pos < nv) clean_at(stg, tile_v0, pos, ck);
            uint32_t eq = 0;
#pragma unroll
            for (int h = 0; h < KPV; ++h) eq += key_at<M>(ck, h) == c;
            uint32_t total;
            const uint32_t incl = block_incl_scan(eq, total);
            uint32_t r = before + incl - eq;
#pragma unroll
            for (int h = 0; h < KPV; ++h) {
                if (key_at<M>(ck, h) == c) {
                    if (r < take) {
                        s->buf_key[first + r] = static_cast<uint16_t>(c);
                        s->buf_idx[first + r] = M::elem(tile_v0 + pos, h);
                    }
                    ++r;
                }
            }
            before += total;
        }
    }

    // The first tile of a CTA's share: a lower bound c on the row's k-th key
    // from the tile's group representatives (one element per group of g, so k
    // distinct elements reach the k-th largest representative), found a byte
    // at a time; g = 1 makes every candidate its own representative (c = the
    // tile's k-th key). The tile then appends its keys > c like any tile; if
    // fewer than k, finish_tile adds its lowest-index keys == c up to k (a
    // crowd of ties at c is never appended whole). Either way the buffer then
    // holds k keys >= c that precede every later key, so later keys need to
    // exceed c.
    __device__ __forceinline__ void first_cut(const uint4 *stg, int64_t tile_v0, int nv) {
        const int tid = threadIdx.x;
        const uint32_t nE = static_cast<uint32_t>(
            M::BLOCK ? nv : min(static_cast<int64_t>(nv) * 8, static_cast<int64_t>(L) - 8 * tile_v0));
        if (nE <= k) {
            count_event(*p, TOPK_CNT_TILE_TAKE_ALL);
            return;
        }
        uint32_t g = 1;
        if (!p->force_direct)
            while (g < static_cast<uint32_t>(M::GMAX) && nE / (4u * g) >= 2u * k) g *= 4u;
        for (;;) {
            PhaseClock clk;
            clk.start(*p);
            // First a window of the 510 keys at and below the largest
            // representative (two keys per bin, the lowest bin holding every
            // lower one; plain atomics: the representatives spread over it).
            // The cut is the lower key of the bin holding the k-th
            // representative; when that bin is crowded (more than k / 4 of
            // them: rows of few distinct values), a count of its upper key
            // makes it exactly the k-th representative, since a key lower by
            // one can be a crowd of its own that later tiles would append.
            uint32_t top = 0;
            rep_walk(stg, tile_v0, nv, g, [&](uint32_t key) { top = max(top, key); });
            top = __reduce_max_sync(0xFFFFFFFFu, top);
            if (lane_id() == 0) s->red[parity][tid >> 5] = top;
            __syncthreads();
#pragma unroll
            for (int w = 0; w < WARPS; ++w) top = max(top, s->red[parity][w]);
            parity ^= 1u;
            if (top != 0u) {
                rep_walk(stg, tile_v0, nv, g, [&](uint32_t key) {
                    if (key) atomicAdd(&s->hwin[2][255u - min((top - key) >> 1, 255u)], 1u);
                });
                __syncthreads();
                uint32_t b, wabove, wtotal;
                const bool ok = find_bin256(s->hwin[2], k, b, wabove, wtotal);
                const uint32_t in_bin = ok ? s->hwin[2][b] : 0u;
                __syncthreads();
                s->hwin[2][tid] = 0u;
                __syncthreads();
                if (ok && b > 0u) {
                    const uint32_t upper = top - 2u * (255u - b);  // bin b: keys upper - 1, upper
                    uint32_t c = upper > 1u ? upper - 1u : 1u;
                    if (in_bin > k / 4u) {
                        uint32_t mine = 0;
                        rep_walk(stg, tile_v0, nv, g, [&](uint32_t key) { mine += key == upper; });
                        uint32_t ups;
                        block_incl_scan(mine, ups);
                        if (wabove + ups >= k) c = upper;
                    }
                    count_event(*p, g == 1u ? TOPK_CNT_TILE_EXACT : TOPK_CNT_TILE_SAMPLED);
                    first_c = c;
                    thr = max(thr, c + 1u);
                    publish(c);
                    clk.stop(*p, TOPK_CNT_CYC_CUT);
                    return;
                }
            }
            rep_pass(stg, tile_v0, nv, g, ALL);
            __syncthreads();
            clk.stop(*p, TOPK_CNT_CYC_REPS);
            clk.start(*p);
            // Every warp reads the same histograms and finds the same bins.
            uint32_t hb, habove, NR;
            if (!find_bin256(s->hwin[2], k, hb, habove, NR)) {
                __syncthreads();
                s->hwin[2][tid] = 0u;
                __syncthreads();
                if (g > 1u) {  // the representatives cannot bound the row: every key its own
                    count_event(*p, TOPK_CNT_TILE_UNBOUNDED);
                    g = 1u;
                    continue;
                }
                count_event(*p, TOPK_CNT_TILE_TAKE_ALL);  // fewer than k candidates here
                return;
            }
            rep_pass(stg, tile_v0, nv, g, hb);
            __syncthreads();
            uint32_t lb, labove, ltotal;
            find_bin256(s->hwin[3], k - habove, lb, labove, ltotal);
            const uint32_t c = (hb << 8) | lb;
            __syncthreads();  // both histograms read: zero them (filter_tile's barriers order it)
            s->hwin[2][tid] = 0u;
            s->hwin[3][tid] = 0u;
            count_event(*p, g == 1u ? TOPK_CNT_TILE_EXACT : TOPK_CNT_TILE_SAMPLED);
            first_c = c;
            thr = max(thr, c + 1u);
            publish(c);
            clk.stop(*p, TOPK_CNT_CYC_CUT);
            return;
        }
    }

    // Keep the buffer entries [0, n) that are selected (key > T, or key == T
    // with index <= cut) at the front of the buffer, in any order. Returns how
    // many were kept.
    __device__ __forceinline__ uint32_t keep_selected(uint32_t n, uint32_t T, uint32_t cut) {
        const int tid = threadIdx.x;
        const uint32_t lt = (1u << lane_id()) - 1u;
        constexpr int PER = 8;
        __syncthreads();
        if (tid == 0) s->v_emit = 0u;
        __syncthreads();
        for (uint32_t base = 0; base < n; base += THREADS * PER) {
            uint32_t key[PER], idx[PER];
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                const uint32_t i = base + static_cast<uint32_t>(e) * THREADS + tid;
                key[e] = i < n ? s->buf_key[i] : 0u;
                idx[e] = i < n ? s->buf_idx[i] : 0u;
            }
            __syncthreads();  // this chunk is read before it is overwritten
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                const bool sel = key[e] != 0u && (key[e] > T || (key[e] == T && idx[e] <= cut));
                const uint32_t b = __ballot_sync(0xFFFFFFFFu, sel);
                const uint32_t at = warp_reserve(&s->v_emit, __popc(b)) + __popc(b & lt);
                if (sel) {
                    s->buf_key[at] = static_cast<uint16_t>(key[e]);
                    s->buf_idx[at] = idx[e];
                }
            }
        }
        __syncthreads();
        return s->v_emit;
    }

    // Write the selected buffer entries [0, n) to out[row, offset + slot]: every
    // key > T, and the `take` lowest-index keys == T (ties beyond TIECAP go
    // through the index radix). Returns the number written.
    __device__ __forceinline__ uint32_t emit_selected(uint32_t n, uint32_t T, uint32_t take, uint32_t offset) {
        const int tid = threadIdx.x;
        const uint32_t lt = (1u << lane_id()) - 1u;
        int32_t *orow = p->out + static_cast<int64_t>(row) * k + offset;
        __syncthreads();
        if (tid == 0) {
            s->v_emit = 0u;
            s->v_ntie = 0u;
        }
        __syncthreads();
        for (uint32_t i0 = 0; i0 < n; i0 += THREADS) {
            const uint32_t i = i0 + tid;
            const uint32_t key = i < n ? s->buf_key[i] : 0u;
            const bool gt = key > T, tie = take && key == T;
            const uint32_t bg = __ballot_sync(0xFFFFFFFFu, gt), bt = __ballot_sync(0xFFFFFFFFu, tie);
            const uint32_t ag = warp_reserve(&s->v_emit, __popc(bg)) + __popc(bg & lt);
            const uint32_t at = warp_reserve(&s->v_ntie, __popc(bt)) + __popc(bt & lt);
            if (gt) orow[ag] = transform(*p, row, static_cast<int32_t>(s->buf_idx[i]));
            if (tie && at < static_cast<uint32_t>(TIECAP)) s->tie_idx[at] = s->buf_idx[i];
        }
        __syncthreads();
        const uint32_t ngt = s->v_emit, e = s->v_ntie;
        if (take == 0u) return ngt;
        if (e <= static_cast<uint32_t>(TIECAP)) {
            if (static_cast<uint32_t>(tid) < e) {
                const uint32_t mine = s->tie_idx[tid];
                uint32_t r = 0;
                if (take < e)
                    for (uint32_t u = 0; u < e; ++u) r += s->tie_idx[u] < mine;
                else
                    r = static_cast<uint32_t>(tid);
                if (r < take) orow[ngt + r] = transform(*p, row, static_cast<int32_t>(mine));
            }
            return ngt + min(take, e);
        }
        // Many ties: cut by index, then write the ties at or below the cut.
        const uint32_t cut = take >= e ? ALL : tie_radix(n, T, take);
        if (tid == 0) s->v_ntie = 0u;
        __syncthreads();
        for (uint32_t i0 = 0; i0 < n; i0 += THREADS) {
            const uint32_t i = i0 + tid;
            const bool sel = i < n && s->buf_key[i] == T && s->buf_idx[i] <= cut;
            const uint32_t b = __ballot_sync(0xFFFFFFFFu, sel);
            const uint32_t at = warp_reserve(&s->v_ntie, __popc(b)) + __popc(b & lt);
            if (sel) orow[ngt + at] = transform(*p, row, static_cast<int32_t>(s->buf_idx[i]));
        }
        return ngt + min(take, e);
    }

    // The largest key of buffer entries [0, n) (0 for none), in every thread.
    __device__ __forceinline__ uint32_t buffer_max(uint32_t n) {
        uint32_t m = 0;
        for (uint32_t i = threadIdx.x; i < n; i += THREADS) m = max(m, static_cast<uint32_t>(s->buf_key[i]));
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        __syncthreads();
        if (threadIdx.x == 0) s->v_bufmax = 0u;
        __syncthreads();
        if (lane_id() == 0 && m) atomicMax(&s->v_bufmax, m);
        __syncthreads();
        return s->v_bufmax;
    }

    // Reduce the buffer to its exact top-k. strict: every buffered key precedes
    // every key still to come, so later keys equal to the cut are dropped too.
    __device__ __forceinline__ void compact(bool strict) {
        const int tid = threadIdx.x;
        __syncthreads();
        const uint32_t n = min(s->v_count, static_cast<uint32_t>(CAP));
        if (n <= k) return;
        // The buffer is about to change: the running histogram is dropped (its
        // words are also the index radix's scratch), rebuilt by the next tile.
        s->hwin[1][tid] = 0u;
        run_ok = false;
        count_event(*p, TOPK_CNT_COMPACTIONS);
        PhaseClock clk;
        clk.start(*p);
        uint32_t T, above;
        window_select(0, n, buf_lo, max(buffer_max(n), buf_lo), k, &T, &above);
        const uint32_t take = k - above;
        const uint32_t cut = tie_cut(n, T, take);
        const uint32_t kept = keep_selected(n, T, cut);
        if (tid == 0) s->v_count = kept;
        buf_lo = T;
        thr = max(thr, strict ? T + 1u : T);
        publish(T);
        __syncthreads();
        clk.stop(*p, TOPK_CNT_CYC_COMPACT);
    }

    // A later tile: append every key >= the threshold.
    //
    // The threshold also rises after every tile: the running histogram of the
    // buffer gives its k-th largest key F, and k keys >= F precede every later
    // key of this CTA's share, so a later key equal to F can no longer be
    // selected (ties go to the lowest index): keep keys >= F + 1 from now on,
    // and tell the peers that the row's k-th key is at least F.
    __device__ __forceinline__ void filter_tile(const uint4 *stg, int64_t tile_v0, int nv) {
        const int tid = threadIdx.x;
        PhaseClock clk;
        clk.start(*p);
        const uint32_t raised = s->v_newthr;  // written before the barrier that ended the last tile
        if (raised > thr) {
            thr = raised;
            best_T = max(best_T, raised - 1u);
            if (raised - 1u >= run_lo + 255u) {  // past the histogram's window: rebuild it
                s->hwin[1][tid] = 0u;
                run_ok = false;
                __syncthreads();
            }
        }
        // Compact ahead of a full buffer only (a refill covers the rest).
        if (s->v_count > static_cast<uint32_t>(3 * CAP / 4) && s->v_count > 2u * k) compact(true);
        if (!run_ok) {
            // Every buffer key >= thr - 1 into the (zero) running histogram,
            // before any append of this tile changes the count.
            run_lo = thr - 1u;
            const uint32_t n = s->v_count;
            for (uint32_t i = tid; i < n; i += THREADS) {
                const uint32_t key = s->buf_key[i];
                if (key >= run_lo) atomicAdd(&s->hwin[1][min(key - run_lo, 255u)], 1u);
            }
            run_ok = true;
            __syncthreads();
        }
        const uint32_t lim = effective_thr();
        // v_full[tpar] and v_arrive[tpar] were zeroed during the last tile; the
        // other words, last read before the barrier that ended the last tile,
        // are zeroed now for the next one.
        tpar ^= 1u;
        if (tid == 0) {
            s->v_full[tpar ^ 1u] = 0u;
            s->v_arrive[tpar ^ 1u] = 0u;
        }
        const bool fast = !M::BLOCK && lim >= 0x8000u && lim <= KEY_POS_INF;
        mask_tail(stg, tile_v0, nv);
        clk.stop(*p, TOPK_CNT_CYC_F_PREP);
        clk.start(*p);
        const uint32_t Q = fast ? build_queue_fast(stg, nv, static_cast<int32_t>(lim) - 0x8000)
                                : build_queue(stg, tile_v0, nv, lim);
        clk.stop(*p, TOPK_CNT_CYC_F_QUEUE);
        clk.start(*p);
        const uint32_t next = fast ? append_fast(stg, tile_v0, Q, 0, lim) : append_keys(stg, tile_v0, Q, 0, lim);
        buf_lo = min(buf_lo, lim);
        f_Q = Q;
        f_next = next;
        f_lim = lim;
        f_fast = fast;
        if (next < Q && lane_id() == 0) s->v_full[tpar] = 1u;
        clk.stop(*p, TOPK_CNT_CYC_F_APPEND);
        clk.start(*p);
        // The first warp done appending finds the buffer's k-th key F for the
        // next tiles while the others still append: each count it reads is at
        // most the number of buffer keys in its bin, so at least k buffer keys
        // are >= F whatever it reads. (The next tile's threshold is raised to
        // F + 1; see above.)
        uint32_t order = 0;
        if (lane_id() == 0) order = atomicAdd(&s->v_arrive[tpar], 1u);
        order = __shfl_sync(0xFFFFFFFFu, order, 0);
        if (order == 0u && run_ok) {
            uint32_t b, above, total;
            if (find_bin256(s->hwin[1], k, b, above, total)) {
                const uint32_t F = run_lo + b;
                if (lane_id() == 0) s->v_newthr = F + 1u;
                publish_lane(F);
            }
        }
        clk.stop(*p, TOPK_CNT_CYC_F_FIND);
    }

    // After the barrier that ends a filter tile: if a warp found the buffer
    // full, compact it and append the rest of the tile (the rest may still tie
    // with the buffer, so the compaction keeps keys equal to its cut).
    __device__ __forceinline__ void finish_tile(const uint4 *stg, int64_t tile_v0, int nv) {
        if (first_c) {
            const uint32_t c = first_c;
            first_c = 0;
            const uint32_t n = s->v_count;  // the keys > c of the first tile (no refill: n <= CAP)
            if (n < k && s->v_full[tpar] == 0u) {
                count_event(*p, TOPK_CNT_TIE_FILLS);
                ordered_ties(stg, tile_v0, nv, c, k - n, n);
                __syncthreads();
                if (threadIdx.x == 0) {
                    s->v_count = k;
                }
                buf_lo = min(buf_lo, c);
                s->hwin[1][threadIdx.x] = 0u;  // rebuilt by the next tile with the ties
                run_ok = false;
                __syncthreads();
                return;
            }
        }
        if (s->v_full[tpar] == 0u) return;  // uniform; rare
        const int tid = threadIdx.x;
        uint32_t next = f_next;
        for (int refill = 0;; ++refill) {
            if (refill == 64) {  // each refill frees >= CAP - k slots: cannot happen
                if (tid == 0) atomicOr(&g_device_status, ERR_BOUNDS);
                break;
            }
            count_event(*p, TOPK_CNT_REFILLS);
            compact(false);
            const uint32_t lim = max(f_lim, thr);  // the buffer now holds k keys >= thr
            next = f_fast ? append_fast(stg, tile_v0, f_Q, next, lim) : append_keys(stg, tile_v0, f_Q, next, lim);
            if (tid == 0) s->v_flag = 0u;
            __syncthreads();
            if (next < f_Q && lane_id() == 0) s->v_flag = 1u;
            __syncthreads();
            if (s->v_flag == 0u) break;  // uniform
        }
    }

    // C == 1: the buffer holds the row's candidates; write its top-k.
    __device__ __forceinline__ void emit_single() {
        s->hwin[1][threadIdx.x] = 0u;  // the index radix's scratch (ordered by the barriers below)
        run_ok = false;
        __syncthreads();
        const uint32_t n = s->v_count;
        uint32_t T = 0, take = 0;
        if (n > k) {
            uint32_t above;
            window_select(0, n, buf_lo, max(buffer_max(n), buf_lo), k, &T, &above);
            take = k - above;
        }
        const uint32_t written = emit_selected(n, T, take, 0);
        int32_t *orow = p->out + static_cast<int64_t>(row) * k;
        for (uint32_t i = written + threadIdx.x; i < k; i += THREADS) orow[i] = -1;
    }

    // Cluster merge: the C buffers (each its CTA's top-k) give the row's k-th
    // key; ties at it go to the lowest indices, lower-ranked CTAs first.
    __device__ __forceinline__ void merge_and_emit() {
        const int tid = threadIdx.x;
        count_event(*p, TOPK_CNT_CLUSTER_MERGES);
        if (s->v_newthr) best_T = max(best_T, s->v_newthr - 1u);  // the last tile's find
        s->hwin[1][tid] = 0u;  // the index radix's scratch
        run_ok = false;
        // The whole buffer takes part (no compaction first): entries below the
        // row's bound are skipped by the histograms and never selected.
        __syncthreads();
        const uint32_t n = min(s->v_count, static_cast<uint32_t>(CAP));
        const uint32_t my_max = buffer_max(n);
        if (tid == 0) {
            atomicMax(&s->shared_thr[slot], best_T);
            atomicMax(&s->shared_max[slot], my_max);
        }
        if (tid < static_cast<int>(C) && tid != static_cast<int>(rank)) {
            red_max_peer(peer_addr(&s->shared_thr[slot], tid), best_T);
            red_max_peer(peer_addr(&s->shared_max[slot], tid), my_max);
        }
        cluster_arrive();
        cluster_wait();
        // Every publication for this row came before the barrier: all threads
        // read the same words.
        const uint32_t LB = max(volatile_load(&s->shared_thr[slot]), 1u);
        const uint32_t HI = volatile_load(&s->shared_max[slot]);
        const uint32_t range = HI > LB ? HI - LB : 0u;
        const int shift = range < 256u ? 0 : (32 - __clz(static_cast<int>(range))) - 8;
        for (uint32_t i = tid; i < n; i += THREADS) {
            const uint32_t key = s->buf_key[i];
            if (key >= LB && HI >= LB) atomicAdd(&s->h_merge[0][window_bin(key, LB, shift)], 1u);
        }
        cluster_arrive();
        cluster_wait();
        {
            uint32_t all, pre;
            cluster_sum(&s->h_merge[0][tid], C, rank, all, pre);
            s->m_all[tid] = all;
            s->m_pre[0][tid] = pre;
        }
        __syncthreads();
        uint32_t b1, above1, total;
        const bool enough = find_bin256(s->m_all, k, b1, above1, total);
        uint32_t T = 0, take = 0, gt_prev = 0, eq_prev = 0, b2 = 0;
        const uint32_t lane = lane_id();
        if (!enough) {
            // Fewer than k candidates in the row: all of them.
            uint32_t x = 0;
            for (uint32_t b = lane; b < 256u; b += 32u) x += s->m_pre[0][b];
            gt_prev = __reduce_add_sync(0xFFFFFFFFu, x);
        } else if (shift == 0) {
            T = LB + b1;
            take = k - above1;
            uint32_t x = 0;
            for (uint32_t b = lane; b < 256u; b += 32u) x += b > b1 ? s->m_pre[0][b] : 0u;
            gt_prev = __reduce_add_sync(0xFFFFFFFFu, x);
            eq_prev = s->m_pre[0][b1];
        } else {
            const uint32_t mask = (1u << shift) - 1u;
            for (uint32_t i = tid; i < n; i += THREADS) {
                const uint32_t key = s->buf_key[i];
                if (key >= LB && ((key - LB) >> shift) == b1) atomicAdd(&s->h_merge[1][(key - LB) & mask], 1u);
            }
            cluster_arrive();
            cluster_wait();
            uint32_t all, pre;
            cluster_sum(&s->h_merge[1][tid], C, rank, all, pre);
            s->m_all[tid] = all;
            s->m_pre[1][tid] = pre;
            __syncthreads();
            uint32_t above2, tot2;
            find_bin256(s->m_all, k - above1, b2, above2, tot2);
            T = LB + (b1 << shift) + b2;
            take = k - above1 - above2;
            uint32_t x = 0;
            for (uint32_t b = lane; b < 256u; b += 32u)
                x += (b > b1 ? s->m_pre[0][b] : 0u) + (b > b2 ? s->m_pre[1][b] : 0u);
            gt_prev = __reduce_add_sync(0xFFFFFFFFu, x);
            eq_prev = s->m_pre[1][b2];
        }
        cluster_arrive();  // done reading the peers' shared memory
        // This CTA's part: keys > T, and its quota of the lowest-index ties.
        const uint32_t quota = take > eq_prev ? take - eq_prev : 0u;
        const uint32_t offset = gt_prev + min(eq_prev, take);
        if (!enough) {
            emit_selected(n, LB - 1u, 0u, offset);  // every key >= LB
        } else {
            emit_selected(n, T, quota, offset);
        }
        const uint32_t selected_total = enough ? k : total;
        int32_t *orow = p->out + static_cast<int64_t>(row) * k;
        for (uint32_t i = selected_total + rank + static_cast<uint32_t>(tid) * C; i < k; i += THREADS * C)
            orow[i] = -1;
        cluster_wait();
        // Every peer is done with this row's shared words: reset them for the
        // row after next (the next row uses the other parity).
        s->h_merge[0][tid] = 0u;
        s->h_merge[1][tid] = 0u;
        if (tid == 0) {
            s->shared_thr[slot] = 0u;
            s->shared_max[slot] = 0u;
        }
    }
};

// Thread 0's view of the tiles still to issue: rows of this cluster in turn,
// each row's share of this CTA in stages of TILE_VEC vectors.
struct Feed {
    int32_t row;
    int32_t tile, ntiles;
    int64_t v0, v1;
};

__device__ __forceinline__ bool row_share(const Params &p, bool block, int32_t row, uint32_t C,
                                          uint32_t rank, int32_t &L, int64_t &V, int64_t &v0,
                                          int64_t &v1) {
    L = min(max(__ldg(p.valid_len + row), 0), p.width);
    const int32_t n = block ? (L + 7) >> 3 : L;
    V = (static_cast<int64_t>(L) + 7) >> 3;
    v0 = V * rank / C;
    v1 = V * (rank + 1) / C;
    return n > p.k;  // false: the row takes 0 .. n-1 without reading logits
}

__device__ __forceinline__ void feed_seek(Feed &f, const Params &p, bool block, int32_t row,
                                          int32_t step, uint32_t C, uint32_t rank) {
    for (; row < p.rows; row += step) {
        int32_t L;
        int64_t V, v0, v1;
        if (row_share(p, block, row, C, rank, L, V, v0, v1) && v1 > v0) {
            f.row = row;
            f.tile = 0;
            f.ntiles = static_cast<int32_t>((v1 - v0 + TILE_VEC - 1) / TILE_VEC);
            f.v0 = v0;
            f.v1 = v1;
            return;
        }
    }
    f.row = p.rows;
}

template <class S>
__device__ __forceinline__ void feed_issue(Feed &f, S &s, int st, const Params &p, bool block,
                                           int32_t step, uint32_t C, uint32_t rank) {
    const int64_t b = f.v0 + static_cast<int64_t>(f.tile) * TILE_VEC;
    const int64_t nvb = f.v1 - b < TILE_VEC ? f.v1 - b : TILE_VEC;
    const uint32_t bytes = static_cast<uint32_t>(nvb * 16);
    const uint4 *src = reinterpret_cast<const uint4 *>(p.logits + static_cast<int64_t>(f.row) * p.row_stride) + b;
    mbar_expect_tx(&s.full[st], bytes);
    bulk_load(&s.stage[st][0], src, bytes, &s.full[st]);
    if (++f.tile == f.ntiles) feed_seek(f, p, block, f.row + step, step, C, rank);
}

template <class M, int NSTAGE, int CAP>
__global__ void __launch_bounds__(THREADS, NSTAGE <= 2 ? 2 : 1) topk_kernel(const Params p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    using S = Smem<NSTAGE, CAP>;
    S &s = *reinterpret_cast<S *>(smem_raw);
    const int tid = threadIdx.x;
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int32_t cid = static_cast<int32_t>(blockIdx.x / C);
    const int32_t ncl = static_cast<int32_t>(gridDim.x / C);

    // Shared-memory set-up first: it touches no global memory, so it overlaps
    // the previous kernel's tail under programmatic dependent launch.
    if (tid == 0) {
        for (int i = 0; i < NSTAGE; ++i) mbar_init(&s.full[i], 1);
        fence_mbar_init();
        s.shared_thr[0] = s.shared_thr[1] = 0u;
        s.shared_max[0] = s.shared_max[1] = 0u;
        s.thr_snap = 0u;
        s.abort_flag = 0u;
    }
    for (int i = 0; i < 4; ++i) s.hwin[i][tid] = 0u;
    s.h_merge[0][tid] = s.h_merge[1][tid] = 0u;
    __syncthreads();
    grid_dependency_wait();
    if (p.release) grid_dependents_release();
    Feed feed;
    if (tid == 0) {
        feed_seek(feed, p, M::BLOCK, cid, ncl, C, rank);
        for (int i = 0; i < NSTAGE && feed.row < p.rows; ++i) feed_issue(feed, s, i, p, M::BLOCK, ncl, C, rank);
    }
    if (C > 1) {
        // Every CTA of the cluster has started and zeroed its shared words
        // before any distributed shared memory access.
        cluster_arrive();
        cluster_wait();
    }

    const Params prm = p;
    Cta<M, NSTAGE, CAP> cta;
    cta.s = &s;
    cta.p = &prm;
    cta.C = C;
    cta.rank = rank;
    cta.k = static_cast<uint32_t>(p.k);
    uint32_t seq = 0, it = 0;
    for (int32_t row = cid; row < p.rows; row += ncl, ++it) {
        int32_t L;
        int64_t V, v0, v1;
        if (!row_share(p, M::BLOCK, row, C, rank, L, V, v0, v1)) {
            // At most k elements: 0 .. n-1, then -1, without reading the logits.
            const int32_t n = M::BLOCK ? (L + 7) >> 3 : L;
            if (rank == 0) count_event(p, TOPK_CNT_BYPASS_ROWS);
            const int32_t lo = static_cast<int32_t>(static_cast<int64_t>(p.k) * rank / C);
            const int32_t hi = static_cast<int32_t>(static_cast<int64_t>(p.k) * (rank + 1) / C);
            for (int32_t i = lo + tid; i < hi; i += THREADS)
                p.out[static_cast<int64_t>(row) * p.k + i] = i < n ? transform(p, row, i) : -1;
            continue;
        }
        cta.row = row;
        cta.L = L;
        cta.V = V;
        cta.thr = M::KMIN;
        cta.buf_lo = 0xFFFFu;
        cta.best_T = 0;
        cta.slot = it & 1u;
        cta.run_ok = false;
        if (tid == 0) {
            s.v_count = 0u;
            s.v_bufmax = 0u;
            s.v_newthr = 0u;
            s.v_full[0] = s.v_full[1] = 0u;
            s.v_arrive[0] = s.v_arrive[1] = 0u;
        }
        s.hwin[1][tid] = 0u;
        cta.snapshot_shared();
        __syncthreads();
        const int ntiles = static_cast<int>((v1 - v0 + TILE_VEC - 1) / TILE_VEC);
        for (int i = 0; i < ntiles; ++i, ++seq) {
            const int st = static_cast<int>(seq % NSTAGE);
            const int64_t tile_v0 = v0 + static_cast<int64_t>(i) * TILE_VEC;
            const int nv = static_cast<int>(v1 - tile_v0 < TILE_VEC ? v1 - tile_v0 : TILE_VEC);
            PhaseClock clk;
            clk.start(p);
            mbar_wait(&s.full[st], (seq / NSTAGE) & 1u, &s.abort_flag);
            clk.stop(p, TOPK_CNT_CYC_WAIT);
            count_event(p, TOPK_CNT_ROUNDS);
            clk.start(p);
            const uint4 *stg = s.stage[st];
            if (i == 0) {
                cta.thr = max(cta.thr, cta.effective_thr());
                cta.first_cut(stg, tile_v0, nv);
                clk.stop(p, TOPK_CNT_CYC_SELECT);
                clk.start(p);
            }
            cta.filter_tile(stg, tile_v0, nv);
            clk.stop(p, TOPK_CNT_CYC_FILTER);
            clk.start(p);
            cta.snapshot_shared();
            __syncthreads();  // every warp is done with this stage (but for a refill)
            cta.finish_tile(stg, tile_v0, nv);
            if (tid == 0 && feed.row < p.rows) {
                fence_proxy_async();
                feed_issue(feed, s, st, p, M::BLOCK, ncl, C, rank);
            }
            clk.stop(p, TOPK_CNT_CYC_F_LOOP);
        }
        PhaseClock fin;
        fin.start(p);
        if (C == 1) {
            cta.emit_single();
        } else {
            cta.merge_and_emit();
        }
        __syncthreads();
        fin.stop(p, TOPK_CNT_CYC_FINISH);
    }
}

// --------------------------------------------- resident-keys (direct) kernel
//
// Rows split over a cluster whose shares fit in shared memory as keys: the
// DecodeTopK page's direct path, with its sample-based cutoff taken from
// representatives. Each CTA streams its share through the stage ring once and
// keeps one 16-bit key per element (0: not a candidate); no candidate buffer,
// no threshold, no compaction. While the tiles stream in, every thread keeps the
// largest key it saw in each tile (a representative) and adds its high byte to
// a histogram. The row's k-th largest representative c (two cluster-wide 8-bit
// passes over the representatives) is a lower bound of the k-th largest key:
// at least k groups hold a key >= c. Only keys >= c (a few per cent) go on: a
// cluster-wide histogram of key - c finds the exact k-th key, and every CTA
// writes its own selected indices from its list of those keys. The exact
// fallback (two 8-bit radix passes over every key) takes the rows where the
// representatives cannot bound the k-th key. Used where a buffer would churn:
// block rows, whose k is large next to a CTA's share.

namespace direct {

constexpr int NT = 256;
constexpr int NSTAGE = 2;
constexpr int RES = 16384;                   // resident keys per CTA
constexpr int MAX_TILES = RES / TILE_VEC;    // stages per share (block rows; token rows take one)
constexpr int LIST_CAP = 1280;               // keys >= the cut listed per CTA (more: emitted by a scan)

struct alignas(128) Smem {
    uint4 stage[NSTAGE][TILE_VEC];
    alignas(16) uint16_t key[RES];           // the share's element keys, in index order
    alignas(16) uint32_t h[3][256];          // this CTA's histograms of the row (peers read them):
                                             // representatives' high / low bytes (or the exact
                                             // passes' keys), then keys - cut
    uint32_t all[256];                       // a histogram summed over the cluster
    uint32_t pre[2][256];                    // ... over the lower-ranked CTAs
    uint16_t rep[MAX_TILES * NT];            // the representative of each thread and tile
    uint32_t list[LIST_CAP];                 // local index << 16 | key, for keys >= the cut
    uint32_t n_list, cursor[2];
    uint32_t red[2][NT / 32];
    uint32_t abort_flag;
    unsigned long long full[NSTAGE];
};
// Two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA.
static_assert(sizeof(Smem) + 1024 <= 233472 / 2, "two resident-keys CTAs must fit on an SM");

template <class M>
struct Share {
    Smem &s;
    const Params &p;
    uint32_t C = 1, rank = 0, par = 0;
    int32_t row = 0, L = 0;
    int64_t V = 0, v0 = 0;
    uint32_t n = 0;  // resident elements

    __device__ Share(Smem &s_, const Params &p_) : s(s_), p(p_) {}

    __device__ __forceinline__ uint32_t block_incl_scan(uint32_t x, uint32_t &total) {
        const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
        const uint32_t inc = warp_incl_scan(x);
        if (lane == 31) s.red[par][warp] = inc;
        __syncthreads();
        const uint32_t w = lane < NT / 32 ? s.red[par][lane] : 0u;
        const uint32_t wi = warp_incl_scan(w);
        total = __shfl_sync(0xFFFFFFFFu, wi, 31);
        const uint32_t pre = __shfl_sync(0xFFFFFFFFu, wi - w, warp);
        par ^= 1u;
        return pre + inc;
    }

    // The keys of one tile's vectors, at their element positions in the share;
    // the thread's largest key of the tile becomes its representative, whose
    // high byte goes into the representatives' histogram h[0].
    __device__ __forceinline__ void keep_tile(const uint4 *stg, int64_t tile_v0, int nv, int tile) {
        uint32_t best = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int pos = j * NT + static_cast<int>(threadIdx.x);
            if (pos >= nv) break;
            const int64_t v = tile_v0 + pos;
            const uint32_t local = static_cast<uint32_t>(v - v0);
            if constexpr (M::BLOCK) {
                const uint32_t key = BlockMode::key(stg[pos], v, V);
                s.key[local] = static_cast<uint16_t>(key);
                best = max(best, key);
            } else {
                uint32_t ck[4];
                TokenMode::clean(stg[pos], v, V, L, ck);  // packed pairs of keys, in element order
                reinterpret_cast<uint4 *>(s.key)[local] = make_uint4(ck[0], ck[1], ck[2], ck[3]);
                best = max(best, umax_halves(umax2(umax2(ck[0], ck[1]), umax2(ck[2], ck[3]))));
            }
        }
        if (!p.force_direct) {  // (uniform: the exact passes start from an empty h[0])
            s.rep[tile * NT + static_cast<int>(threadIdx.x)] = static_cast<uint16_t>(best);
            agg_add(s.h[0], best >> 8, best != 0u);
        }
    }

    // Every CTA's histogram `which` complete (a cluster barrier), then its sum
    // over the cluster (all) and, for pre_slot >= 0, over the lower ranks.
    __device__ __forceinline__ void gather(int which, int pre_slot) {
        const int tid = threadIdx.x;
        if (C > 1) {
            cluster_arrive();
            cluster_wait();
        } else {
            __syncthreads();
        }
        uint32_t all = s.h[which][tid], pre = 0;
        if (C > 1) cluster_sum(&s.h[which][tid], C, rank, all, pre);
        s.all[tid] = all;
        if (pre_slot >= 0) s.pre[pre_slot][tid] = pre;
        __syncthreads();
    }

    __device__ __forceinline__ void put(int32_t *orow, uint32_t slot, uint32_t local) const {
        const int64_t e = M::BLOCK ? v0 + local : 8 * v0 + local;
        orow[slot] = transform(p, row, static_cast<int32_t>(e));
    }

    // Key h (0..7) of a group of eight packed in a uint4.
    static __device__ __forceinline__ uint32_t key_of(const uint4 &w, int h) {
        const uint32_t x = (h & 4) ? ((h & 2) ? w.w : w.z) : ((h & 2) ? w.y : w.x);
        return (h & 1) ? (x >> 16) : (x & 0xFFFFu);
    }

    // This CTA's keys > T at slots gt_prev + .. (after those of the lower ranks,
    // in any order), then its quota of the lowest-index keys == T at slots
    // G + eq_prev + .. (after those of the lower ranks). Each thread owns a
    // contiguous run of groups, so ties rank in index order by thread, then
    // within the run. ties = false: no key == T is taken.
    __device__ void emit_scan(uint32_t T, uint32_t G, uint32_t gt_prev, uint32_t eq_prev,
                              uint32_t take, bool ties) {
        const int tid = threadIdx.x;
        const uint32_t lane = lane_id();
        const uint32_t groups = (n + 7u) / 8u;
        const uint4 *k4 = reinterpret_cast<const uint4 *>(s.key);
        const uint32_t quota = take > eq_prev ? take - eq_prev : 0u;
        int32_t *orow = p.out + static_cast<int64_t>(row) * p.k;
        const uint32_t run = (groups + NT - 1) / NT;
        const uint32_t g_lo = min(groups, static_cast<uint32_t>(tid) * run);
        const uint32_t g_n = min(groups, g_lo + run) - g_lo;
        uint32_t gt = 0, eq = 0;
        for (uint32_t j = 0; j < g_n; ++j) {
            const uint32_t g = g_lo + (j + lane) % g_n;  // rotated: lanes spread over banks
            const uint4 w = k4[g];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const uint32_t key = key_of(w, h);
                gt += key > T;
                eq += ties && key == T;
            }
        }
        uint32_t tot;
        const uint32_t packed = gt | (eq << 16);
        const uint32_t ex = block_incl_scan(packed, tot) - packed;
        uint32_t rg = gt_prev + (ex & 0xFFFFu);
        if (gt) {
            for (uint32_t j = 0; j < g_n; ++j) {
                const uint32_t g = g_lo + (j + lane) % g_n;
                const uint4 w = k4[g];
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    if (key_of(w, h) > T) put(orow, rg++, 8u * g + static_cast<uint32_t>(h));
            }
        }
        uint32_t re = ex >> 16;
        if (eq && re < quota) {  // in index order
            for (uint32_t j = 0; j < g_n && re < quota; ++j) {
                const uint32_t g = g_lo + j;
                const uint4 w = k4[g];
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    if (key_of(w, h) == T) {
                        if (re < quota) put(orow, G + eq_prev + re, 8u * g + static_cast<uint32_t>(h));
                        ++re;
                    }
                }
            }
        }
    }

    // The exact k-th key from two cluster-wide 8-bit radix passes over every
    // resident key (h[0] and h[1] start empty), then the emission. The keys are
    // read eight at a time (16 bytes, consecutive across lanes); groups past the
    // share read as zero (no candidate). Rows with fewer than k candidates take
    // them all and pad with -1.
    __device__ void exact_select(PhaseClock &clk) {
        const int tid = threadIdx.x;
        const uint32_t k = static_cast<uint32_t>(p.k);
        const uint32_t groups = (n + 7u) / 8u;
        const uint4 *k4 = reinterpret_cast<const uint4 *>(s.key);
        const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
        // Pass 1: high bytes. (Every lane of a warp runs every iteration: the
        // warp-wide match in agg_add needs them all.)
        for (uint32_t g0 = 0; g0 < groups; g0 += NT) {
            const uint32_t g = g0 + static_cast<uint32_t>(tid);
            const uint4 w = g < groups ? k4[g] : zero4;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const uint32_t key = key_of(w, h);
                agg_add(s.h[0], key >> 8, key != 0u);
            }
        }
        gather(0, 0);
        clk.stop(p, TOPK_CNT_CYC_CUT);
        clk.start(p);
        uint32_t b1, above1, total;
        const bool enough = find_bin256(s.all, k, b1, above1, total);
        uint32_t T = 0, take = 0, gt_prev = 0, eq_prev = 0;
        const uint32_t lane = lane_id();
        if (enough) {
            // Pass 2: low bytes of the keys in bin b1 (a warp with none skips the match).
            for (uint32_t g0 = 0; g0 < groups; g0 += NT) {
                const uint32_t g = g0 + static_cast<uint32_t>(tid);
                const uint4 w = g < groups ? k4[g] : zero4;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const uint32_t key = key_of(w, h);
                    const bool in = key != 0u && (key >> 8) == b1;
                    if (__any_sync(0xFFFFFFFFu, in)) agg_add(s.h[1], key & 0xFFu, in);
                }
            }
            gather(1, 1);
            uint32_t b2, above2, tot2;
            find_bin256(s.all, k - above1, b2, above2, tot2);
            T = (b1 << 8) | b2;
            take = k - above1 - above2;
            uint32_t x = 0;
            for (uint32_t b = lane; b < 256u; b += 32u)
                x += (b > b1 ? s.pre[0][b] : 0u) + (b > b2 ? s.pre[1][b] : 0u);
            gt_prev = __reduce_add_sync(0xFFFFFFFFu, x);
            eq_prev = s.pre[1][b2];
        } else {
            // Fewer than k candidates in the row: every one of them.
            uint32_t x = 0;
            for (uint32_t b = lane; b < 256u; b += 32u) x += s.pre[0][b];
            gt_prev = __reduce_add_sync(0xFFFFFFFFu, x);
            T = 0u;  // every key > 0
        }
        if (C > 1) cluster_arrive();  // done reading the peers' histograms
        clk.stop(p, TOPK_CNT_CYC_EXACT);
        clk.start(p);
        emit_scan(T, enough ? k - take : total, gt_prev, eq_prev, take, enough);
        const uint32_t selected = enough ? k : total;
        int32_t *orow = p.out + static_cast<int64_t>(row) * k;
        for (uint32_t i = selected + rank + static_cast<uint32_t>(tid) * C; i < k; i += NT * C) orow[i] = -1;
    }

    // This CTA's keys >= c: listed (local index << 16 | key; past LIST_CAP only
    // counted) and binned by key - c into h[2], the last bin holding every key
    // >= c + 255. A counting pass over the thread's groups (g = j * NT + tid),
    // one reservation per warp, then a writing pass over the groups that hold
    // such keys.
    __device__ __forceinline__ void list_survivors(uint32_t c) {
        constexpr uint32_t GPT = RES / 8 / NT;  // groups per thread, at most
        const uint32_t groups = (n + 7u) / 8u;
        const uint4 *k4 = reinterpret_cast<const uint4 *>(s.key);
        const uint32_t tid = threadIdx.x;
        uint32_t cnt = 0, hold = 0;
#pragma unroll
        for (uint32_t j = 0; j < GPT; ++j) {
            const uint32_t g = j * NT + tid;
            if (g < groups) {
                const uint4 w = k4[g];
                if (umax_halves(umax2(umax2(w.x, w.y), umax2(w.z, w.w))) >= c) {
                    hold |= 1u << j;
#pragma unroll
                    for (int h = 0; h < 8; ++h) cnt += key_of(w, h) >= c;
                }
            }
        }
        const uint32_t inc = warp_incl_scan(cnt);
        uint32_t at = warp_reserve(&s.n_list, __shfl_sync(0xFFFFFFFFu, inc, 31)) + inc - cnt;
        while (hold) {
            const uint32_t j = static_cast<uint32_t>(__ffs(hold) - 1);
            hold &= hold - 1u;
            const uint32_t g = j * NT + tid;
            const uint4 w = k4[g];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const uint32_t key = key_of(w, h);
                if (key >= c) {
                    if (at < static_cast<uint32_t>(LIST_CAP))
                        s.list[at] = ((8u * g + static_cast<uint32_t>(h)) << 16) | key;
                    ++at;
                    atomicAdd(&s.h[2][min(key - c, 255u)], 1u);
                }
            }
        }
    }

    // The selection from the representatives' cut; false (with nothing
    // written) when the row needs the exact passes: fewer than k
    // representatives, or the k-th key in the window's last bin. The answer is
    // the same on every CTA of the cluster (it comes from cluster-wide sums).
    __device__ bool cut_select(uint32_t ntiles, PhaseClock &clk) {
        const int tid = threadIdx.x;
        const uint32_t k = static_cast<uint32_t>(p.k);
        const uint32_t lane = lane_id();
        clk.stop(p, TOPK_CNT_CYC_CUT);
        clk.start(p);
        gather(0, -1);  // the representatives' high bytes
        clk.stop(p, TOPK_CNT_CYC_ALIGN);
        clk.start(p);
        // Past that barrier no thread uses the previous row's list: reset it
        // (the next barrier publishes the zeros).
        if (tid == 0) s.n_list = s.cursor[0] = s.cursor[1] = 0u;
        uint32_t b1, above1, total;
        if (!find_bin256(s.all, k, b1, above1, total)) {
            if (rank == 0) count_event(p, TOPK_CNT_TILE_UNBOUNDED);
            return false;
        }
        // The low bytes of the representatives in bin b1.
        for (uint32_t j = 0; j < ntiles; ++j) {
            const uint32_t r = s.rep[j * NT + static_cast<uint32_t>(tid)];
            const bool in = r != 0u && (r >> 8) == b1;
            if (__any_sync(0xFFFFFFFFu, in)) agg_add(s.h[1], r & 0xFFu, in);
        }
        gather(1, -1);
        uint32_t b2, above2, tot2;
        find_bin256(s.all, k - above1, b2, above2, tot2);
        const uint32_t c = (b1 << 8) | b2;  // the row's k-th largest representative
        clk.stop(p, TOPK_CNT_CYC_CUT);
        clk.start(p);
        list_survivors(c);
        gather(2, 0);
        clk.stop(p, TOPK_CNT_CYC_SURVIVORS);
        clk.start(p);
        uint32_t t, above, tot3;
        find_bin256(s.all, k, t, above, tot3);  // at least k keys are >= c
        if (t == 255u) {  // the k-th key is >= c + 255: not resolved by the window
            if (rank == 0) count_event(p, TOPK_CNT_TILE_OVERFLOW);
            return false;
        }
        if (rank == 0) count_event(p, TOPK_CNT_TILE_SAMPLED);
        const uint32_t T = c + t;       // the row's k-th largest key
        const uint32_t take = k - above;  // keys == T to take, lowest indices first
        uint32_t x = 0;
        for (uint32_t b = lane; b < 256u; b += 32u) x += b > t ? s.pre[0][b] : 0u;
        const uint32_t gt_prev = __reduce_add_sync(0xFFFFFFFFu, x);
        const uint32_t eq_prev = s.pre[0][t];
        const uint32_t my_eq = s.h[2][t];
        if (C > 1) cluster_arrive();  // done reading the peers' histograms
        clk.stop(p, TOPK_CNT_CYC_EXACT);
        clk.start(p);
        const uint32_t quota = take > eq_prev ? min(take - eq_prev, my_eq) : 0u;
        const uint32_t listed = s.n_list;
        const bool partial = quota != 0u && quota != my_eq;  // some of this CTA's ties, lowest first
        if (listed > static_cast<uint32_t>(LIST_CAP) || (partial && my_eq > static_cast<uint32_t>(NT))) {
            // Listed only in part, or too many ties to rank: from the resident keys.
            emit_scan(T, above, gt_prev, eq_prev, take, true);
            return true;
        }
        // From the list: keys > T at warp-reserved slots (the order within a
        // class is free); keys == T likewise when this CTA takes all of them,
        // else gathered (into pre[1], unused on this path) and ranked by index.
        int32_t *orow = p.out + static_cast<int64_t>(row) * k;
        uint32_t *ties = s.pre[1];
        const uint32_t lt = (1u << lane) - 1u;
        for (uint32_t i0 = 0; i0 < listed; i0 += NT) {
            const uint32_t i = i0 + static_cast<uint32_t>(tid);
            const uint32_t e = i < listed ? s.list[i] : 0u;
            const uint32_t key = e & 0xFFFFu;
            const bool gt = key > T, eq = quota != 0u && key == T;
            const uint32_t bg = __ballot_sync(0xFFFFFFFFu, gt), be = __ballot_sync(0xFFFFFFFFu, eq);
            const uint32_t og = warp_reserve(&s.cursor[0], __popc(bg));
            const uint32_t oe = warp_reserve(&s.cursor[1], __popc(be)) + __popc(be & lt);
            if (gt) put(orow, gt_prev + og + __popc(bg & lt), e >> 16);
            if (eq) {
                if (partial) ties[oe] = e >> 16;
                else put(orow, above + eq_prev + oe, e >> 16);
            }
        }
        if (partial) {
            __syncthreads();
            if (static_cast<uint32_t>(tid) < my_eq) {
                const uint32_t mine = ties[tid];
                uint32_t r = 0;
                for (uint32_t j = 0; j < my_eq; ++j) r += ties[j] < mine;
                if (r < quota) put(orow, above + eq_prev + r, mine);
            }
        }
        return true;
    }

    __device__ void select_and_emit(uint32_t ntiles) {
        const int tid = threadIdx.x;
        PhaseClock clk;
        clk.start(p);
        bool done = false;
        if (!p.force_direct) {
            done = cut_select(ntiles, clk);
            if (!done) {
                // Every peer must be done reading h[0] and h[1] before the exact
                // passes refill them.
                if (C > 1) {
                    cluster_arrive();
                    cluster_wait();
                } else {
                    __syncthreads();
                }
                s.h[0][tid] = 0u;
                s.h[1][tid] = 0u;
                __syncthreads();
                clk.start(p);
            }
        }
        if (!done) {
            if (rank == 0) count_event(p, TOPK_CNT_TILE_EXACT);
            exact_select(clk);
        }
        if (C > 1) cluster_wait();
        else __syncthreads();
        clk.stop(p, TOPK_CNT_CYC_FINISH);
        // Every peer is done with this row's histograms: clear them for the next.
        // (The list and its cursors may still be in use by this CTA's slower
        // warps: the wait above passes once every thread has arrived, which each
        // did before emitting.)
        s.h[0][tid] = 0u;
        s.h[1][tid] = 0u;
        s.h[2][tid] = 0u;
    }
};

template <class M>
__global__ void __launch_bounds__(NT, 2) topk_direct_kernel(const Params p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &s = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x;
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int32_t cid = static_cast<int32_t>(blockIdx.x / C);
    const int32_t ncl = static_cast<int32_t>(gridDim.x / C);
    PhaseClock whole;
    whole.start(p);

    if (tid == 0) {  // (shared-memory set-up before the wait, as in topk_kernel)
        for (int i = 0; i < NSTAGE; ++i) mbar_init(&s.full[i], 1);
        fence_mbar_init();
        s.abort_flag = 0u;
    }
    s.h[0][tid] = s.h[1][tid] = s.h[2][tid] = 0u;
    if (tid == 0) s.n_list = s.cursor[0] = s.cursor[1] = 0u;
    __syncthreads();
    grid_dependency_wait();
    if (p.release) grid_dependents_release();

    Feed feed;
    if (tid == 0) {
        feed_seek(feed, p, M::BLOCK, cid, ncl, C, rank);
        for (int i = 0; i < NSTAGE && feed.row < p.rows; ++i) feed_issue(feed, s, i, p, M::BLOCK, ncl, C, rank);
    }
    if (C > 1) {  // every CTA started and zeroed before any distributed access
        cluster_arrive();
        cluster_wait();
    }
    Share<M> sh(s, p);
    sh.C = C;
    sh.rank = rank;
    uint32_t seq = 0;
    for (int32_t row = cid; row < p.rows; row += ncl) {
        int32_t L;
        int64_t V, v0, v1;
        if (!row_share(p, M::BLOCK, row, C, rank, L, V, v0, v1)) {
            const int32_t n = M::BLOCK ? (L + 7) >> 3 : L;
            if (rank == 0) count_event(p, TOPK_CNT_BYPASS_ROWS);
            const int32_t lo = static_cast<int32_t>(static_cast<int64_t>(p.k) * rank / C);
            const int32_t hi = static_cast<int32_t>(static_cast<int64_t>(p.k) * (rank + 1) / C);
            for (int32_t i = lo + tid; i < hi; i += NT)
                p.out[static_cast<int64_t>(row) * p.k + i] = i < n ? transform(p, row, i) : -1;
            continue;
        }
        sh.row = row;
        sh.L = L;
        sh.V = V;
        sh.v0 = v0;
        sh.n = static_cast<uint32_t>(M::BLOCK ? v1 - v0 : 8 * (v1 - v0));
        const int ntiles = static_cast<int>((v1 - v0 + TILE_VEC - 1) / TILE_VEC);
        for (int i = 0; i < ntiles; ++i, ++seq) {
            const int st = static_cast<int>(seq % NSTAGE);
            const int64_t tile_v0 = v0 + static_cast<int64_t>(i) * TILE_VEC;
            const int nv = static_cast<int>(v1 - tile_v0 < TILE_VEC ? v1 - tile_v0 : TILE_VEC);
            PhaseClock clk;
            clk.start(p);
            mbar_wait(&s.full[st], (seq / NSTAGE) & 1u, &s.abort_flag);
            clk.stop(p, TOPK_CNT_CYC_WAIT);
            count_event(p, TOPK_CNT_ROUNDS);
            clk.start(p);
            sh.keep_tile(s.stage[st], tile_v0, nv, i);
            __syncthreads();  // every thread is done with this stage
            clk.stop(p, TOPK_CNT_CYC_FILTER);
            if (tid == 0 && feed.row < p.rows) {
                fence_proxy_async();
                feed_issue(feed, s, st, p, M::BLOCK, ncl, C, rank);
            }
        }
        if (tid == 0)  // the last group's keys past the share: no candidates
            for (uint32_t i = sh.n; i < ((sh.n + 7u) & ~7u); ++i) s.key[i] = 0u;
        __syncthreads();
        if (rank == 0) count_event(p, TOPK_CNT_DIRECT_ROWS);
        sh.select_and_emit(static_cast<uint32_t>(ntiles));
        __syncthreads();
    }
    whole.stop(p, TOPK_CNT_CYC_KERNEL);
}

}  // namespace direct

// ------------------------------------------------------- one-tile rows kernel
//
// Rows whose valid prefix fits one tile (at most 2048 vectors) take a leaner
// path: 512 threads hold the row in registers (4 vectors each), the stage it
// came through is handed back to the copy ring at once, and the selection runs
// in a handful of barrier phases: representatives -> cut -> survivors -> exact
// cut -> write. Same cutoff argument as the streamed kernel.
namespace one {

// Everything of the one-tile path for a CTA of NT_ threads (256: several CTAs
// per SM for many rows; 512: one, for rows that do not fill the SMs, where a
// row's latency is what counts) with a survivor list of SURV_ entries (2048
// for k <= 1024 fits four CTAs per SM; 4096 for larger k, three).
template <int NT_, int SURV_>
struct Tile {
static constexpr int NT = NT_;
static constexpr int NW = NT / 32;
static constexpr int NV = 2048 / NT;         // vectors per thread
static constexpr int NTILE = NT * NV;        // 2048 vectors
static constexpr int NSTAGE = NT == 256 ? 1 : 2;  // 256: the other CTAs on the SM cover its copies
static constexpr int SURV_CAP = SURV_;
static constexpr int REP_CAP = 4096;         // stored representatives (groups of >= 4 logits)
static constexpr int QN = 32 * NV;           // queue entries of one warp
static constexpr int TAB_CAP = 256;         // page ids of a row staged in shared memory (<= NT)

struct alignas(128) Smem {
    uint4 stage[NSTAGE][NTILE];
    union {                                  // the representatives are done before survivors start
        struct {
            uint32_t surv_idx[SURV_CAP + 4]; // + a spare slot for writes past the end
            uint16_t surv_key[SURV_CAP + 8];
        };
        uint16_t rep[REP_CAP];               // the row's representatives (0 = none)
    };
    alignas(16) uint32_t hs[4][256];         // [0], [1]: the cut's byte passes (zero between
                                             // uses); [2 + row parity]: the row's window
    uint32_t tie_idx[TIECAP];
    uint8_t queue[NW][QN];                   // (j << 5) | lane of queued vectors j * NT + thread
    int32_t tab[TAB_CAP];
    uint32_t red[2][NW];
    uint32_t bc[4];
    uint32_t v_cnt[2];                       // survivor counts, by row parity
    uint32_t v_smax, v_ntie;
    uint32_t abort_flag;
    unsigned long long full[NSTAGE];
};

// Histograms are read and written as 16-byte vectors; stages are bulk-copy targets.
static_assert(offsetof(Smem, hs) % 16 == 0 && offsetof(Smem, stage) % 128 == 0, "shared layout");
static_assert(TAB_CAP <= NT, "one page id per thread");


static __device__ __forceinline__ uint32_t block_scan(Smem &s, uint32_t &par, uint32_t x, uint32_t &total) {
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    const uint32_t inc = warp_incl_scan(x);
    if (lane == 31) s.red[par][warp] = inc;
    __syncthreads();
    const uint32_t w = lane < NW ? s.red[par][lane] : 0u;
    const uint32_t wi = warp_incl_scan(w);
    total = __shfl_sync(0xFFFFFFFFu, wi, 31);
    const uint32_t pre = __shfl_sync(0xFFFFFFFFu, wi - w, warp);
    par ^= 1u;
    return pre + inc;
}

// Warp 0 finds the bin of `hist` holding the q-th largest and zeroes the
// histogram; the caller's __syncthreads then publishes s.bc = {bin, above, total}.
static __device__ __forceinline__ void warp0_find(Smem &s, uint32_t *hist, uint32_t q) {
    if (threadIdx.x < 32) {
        uint32_t b, above, total;
        find_bin256(hist, q, b, above, total);
        reinterpret_cast<uint4 *>(hist)[2 * threadIdx.x] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4 *>(hist)[2 * threadIdx.x + 1] = make_uint4(0, 0, 0, 0);
        if (threadIdx.x == 0) {
            s.bc[0] = b;
            s.bc[1] = above;
            s.bc[2] = total;
        }
    }
}

// The half h (0..7) of a vector as a 16-bit value.
static __device__ __forceinline__ uint32_t half_of(const uint4 &r, int h) {
    const uint32_t w = (h & 4) ? ((h & 2) ? r.w : r.z) : ((h & 2) ? r.y : r.x);
    return (h & 1) ? (w >> 16) : (w & 0xFFFFu);
}

template <class M>
struct Row {
    Smem &s;
    const Params &p;
    uint4 *stg = nullptr;         // the row's vectors, in shared memory
    uint32_t par = 0;
    int32_t row = 0, L = 0, V = 0;
    int32_t *orow = nullptr;      // the row's k output slots
    uint32_t k = 0;
    uint32_t guess = 0;   // the cut carried over from this CTA's previous row (0: none)
    uint32_t rp = 0;      // parity of the rows this CTA has selected
    bool tab = false;     // the row's page ids are in s.tab

    __device__ Row(Smem &s_, const Params &p_) : s(s_), p(p_) {}

    // Vector at position pos: lanes without an element read as 0x8000 (a
    // negative value no cut can select and no group maximum prefers). The
    // row's last vector is masked in place by mask_tail.
    __device__ __forceinline__ uint4 vec(int pos) const {
        if (pos >= V) return make_uint4(0x80008000u, 0x80008000u, 0x80008000u, 0x80008000u);
        return stg[pos];
    }

    // Token mode: overwrite the lanes of the last vector past the valid length
    // with 0x8000, by the thread that owns that position (every later reader of
    // it is that thread or, after a warp barrier, its warp).
    __device__ __forceinline__ void mask_tail() const {
        if (M::BLOCK || (L & 7) == 0 || static_cast<int>(threadIdx.x) != (V - 1) % NT) return;
        const int lanes = L & 7;
        const uint4 r = stg[V - 1];
        uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int h = 0; h < 8; ++h)
            if (h >= lanes)
                w[h >> 1] = (w[h >> 1] & ((h & 1) ? 0x0000FFFFu : 0xFFFF0000u)) |
                            ((h & 1) ? 0x80000000u : 0x00008000u);
        stg[V - 1] = make_uint4(w[0], w[1], w[2], w[3]);
    }

    __device__ __forceinline__ uint32_t bkey(int pos) const {
        return pos < V ? BlockMode::key(stg[pos], pos, V) : 0u;
    }

    __device__ __forceinline__ void clean(int pos, uint32_t (&ck)[4]) const {
        if (pos < V) M::clean(stg[pos], pos, V, L, ck);
        else ck[0] = ck[1] = ck[2] = ck[3] = 0u;
    }

    __device__ __forceinline__ void put(uint32_t slot, uint32_t idx) const {
        int32_t v = static_cast<int32_t>(idx);
        if (tab) v = s.tab[idx >> p.page_shift] * p.block_rows + (v & ((1 << p.page_shift) - 1));
        else v = transform(p, row, v);
        orow[slot] = v;
    }

    // Representatives of groups of G elements of this thread's vectors
    // j * NT + tid (token: G logits, within a vector for G <= 8, else whole
    // vectors; block: G blocks), fed to f(slot, r, key) in a fixed slot order
    // (r: the thread's r-th representative, slot = r * NT + tid).
    template <int G, class F>
    __device__ __forceinline__ void reps(F &&f) const {
        const int tid = threadIdx.x;
        if constexpr (M::BLOCK) {
#pragma unroll
            for (int j = 0; j < NV; j += G) {
                uint32_t acc = 0;
#pragma unroll
                for (int i = 0; i < G; ++i) acc = max(acc, bkey((j + i) * NT + tid));
                f((j / G) * NT + tid, j / G, acc);
            }
        } else if constexpr (G == 4) {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const uint4 r = vec(j * NT + tid);
                f((2 * j) * NT + tid, 2 * j, rep_key(smax_halves(smax2(r.x, r.y)), 1u));
                f((2 * j + 1) * NT + tid, 2 * j + 1, rep_key(smax_halves(smax2(r.z, r.w)), 1u));
            }
        } else {
            constexpr int PER = G / 8;  // whole vectors per group
#pragma unroll
            for (int j = 0; j < NV; j += PER) {
                uint32_t acc = vec_smax(vec(j * NT + tid));
#pragma unroll
                for (int i = 1; i < PER; ++i) acc = smax2(acc, vec_smax(vec((j + i) * NT + tid)));
                f((j / PER) * NT + tid, j / PER, rep_key(smax_halves(acc), 1u));
            }
        }
    }

    // A cut at most the k-th largest representative of groups of G, so that
    // at least k keys are >= it. First a window of the 510 keys at and below
    // the largest representative (two keys per bin, the lowest bin holding
    // everything below): one pass with plain atomics, as the bins are spread;
    // the cut is the lower key of the bin holding the k-th representative.
    // When that bin is the lowest, two byte passes over the stored
    // representatives give it exactly (high byte, then low byte within the
    // high byte's bin). False when there are fewer than k representatives.
    template <int G>
    __device__ __forceinline__ bool rep_cut(uint32_t &c) {
        constexpr int R = M::BLOCK ? NV / G : (G >= 8 ? NV * 8 / G : NV * 2);
        constexpr int NREP = R * NT;
        static_assert(NREP <= REP_CAP, "representatives do not fit");
        uint32_t v[R];
        reps<G>([&](int slot, int r, uint32_t key) {
            s.rep[slot] = static_cast<uint16_t>(key);
            v[r] = key;
        });
        uint32_t top = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) top = max(top, v[r]);
        top = __reduce_max_sync(0xFFFFFFFFu, top);
        if (lane_id() == 0) s.red[par][threadIdx.x >> 5] = top;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < NW; ++w) top = max(top, s.red[par][w]);
        par ^= 1u;
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (v[r] != 0u) atomicAdd(&s.hs[0][255u - min((top - v[r]) >> 1, 255u)], 1u);
        __syncthreads();
        warp0_find(s, s.hs[0], k);
        __syncthreads();
        if (s.bc[2] < k) return false;
        if (s.bc[0] > 0u) {
            c = static_cast<uint32_t>(max(static_cast<int>(top) - 2 * (255 - static_cast<int>(s.bc[0])) - 1, 1));
            return true;
        }
        for (int i = threadIdx.x; i < NREP; i += NT) {
            const uint32_t key = s.rep[i];
            agg_add(s.hs[0], key >> 8, key != 0u);
        }
        __syncthreads();
        warp0_find(s, s.hs[0], k);
        __syncthreads();
        const uint32_t hb = s.bc[0], habove = s.bc[1], nreps = s.bc[2];
        if (nreps < k) return false;
#pragma unroll
        for (int i = threadIdx.x; i < NREP; i += NT) {
            const uint32_t key = s.rep[i];
            agg_add(s.hs[1], key & 0xFFu, key != 0u && (key >> 8) == hb);
        }
        __syncthreads();
        warp0_find(s, s.hs[1], k - habove);
        __syncthreads();
        c = (hb << 8) | s.bc[0];
        return true;
    }

    // The exact path's cut: every candidate key is its own representative.
    __device__ bool exact_cut(uint32_t &c) {
        const int tid = threadIdx.x;
        for (int j = 0; j < NV; ++j) {
            uint32_t ck[4];
            clean(j * NT + tid, ck);
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) {
                const uint32_t key = key_at<M>(ck, h);
                agg_add(s.hs[0], key >> 8, key != 0u);
            }
        }
        __syncthreads();
        warp0_find(s, s.hs[0], k);
        __syncthreads();
        const uint32_t hb = s.bc[0], habove = s.bc[1], nkeys = s.bc[2];
        if (nkeys < k) return false;
        for (int j = 0; j < NV; ++j) {
            uint32_t ck[4];
            clean(j * NT + tid, ck);
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) {
                const uint32_t key = key_at<M>(ck, h);
                agg_add(s.hs[1], key & 0xFFu, key != 0u && (key >> 8) == hb);
            }
        }
        __syncthreads();
        warp0_find(s, s.hs[1], k - habove);
        __syncthreads();
        c = (hb << 8) | s.bc[0];
        return true;
    }

    // Every candidate key its own representative (rows too short for groups):
    // the exact k-th largest key, from a window of the 512 keys at and below
    // the largest key (two keys per bin; the keys in it spread over the bins:
    // plain atomics) and a count of the upper key of the bin that holds it
    // (exact: a crowd of ties at it may be written by index-ordered rescans).
    // When it lies lower, the radix passes of exact_cut; rows that select a
    // quarter of their elements or more go there directly (their k-th key is
    // far below the largest). False when the row has fewer than k candidates.
    __device__ bool window_cut(uint32_t &c) {
        const int tid = threadIdx.x;
        if (4u * k >= static_cast<uint32_t>(M::BLOCK ? V : L)) return exact_cut(c);
        uint32_t top = 0;
        for (int j = 0; j < NV; ++j) {
            uint32_t ck[4];
            clean(j * NT + tid, ck);
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) top = max(top, key_at<M>(ck, h));
        }
        top = __reduce_max_sync(0xFFFFFFFFu, top);
        if (lane_id() == 0) s.red[par][tid >> 5] = top;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < NW; ++w) top = max(top, s.red[par][w]);
        par ^= 1u;
        if (top == 0u) return false;  // no candidate at all
        const uint32_t lo = top > 511u ? top - 511u : 1u;
        for (int j = 0; j < NV; ++j) {
            uint32_t ck[4];
            clean(j * NT + tid, ck);
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) {
                const uint32_t key = key_at<M>(ck, h);
                if (key >= lo) atomicAdd(&s.hs[0][255u - ((top - key) >> 1)], 1u);
            }
        }
        __syncthreads();
        warp0_find(s, s.hs[0], k);
        __syncthreads();
        const uint32_t b = s.bc[0], above_b = s.bc[1], in_window = s.bc[2];
        __syncthreads();  // every thread has read s.bc
        if (in_window < k) return exact_cut(c);
        const uint32_t upper = top - 2u * (255u - b);  // bin b: keys upper - 1 and upper
        uint32_t n_up = 0;
        for (int j = 0; j < NV; ++j) {
            uint32_t ck[4];
            clean(j * NT + tid, ck);
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) n_up += key_at<M>(ck, h) == upper;
        }
        uint32_t ups;
        block_scan(s, par, n_up, ups);
        c = above_b + ups >= k ? upper : upper - 1u;
        return true;
    }

    __device__ __forceinline__ bool cut_for(uint32_t g, uint32_t &c) {
        // (a group is at most a thread's NV vectors)
        if constexpr (M::BLOCK) {
            if constexpr (NV >= 8) if (g == 8u) return rep_cut<8>(c);
            if constexpr (NV >= 4) if (g == 4u) return rep_cut<4>(c);
            if (g == 2u) return rep_cut<2>(c);
            return p.force_direct ? exact_cut(c) : window_cut(c);
        } else {
            if constexpr (NV >= 8) if (g == 64u) return rep_cut<64>(c);
            if constexpr (NV >= 4) if (g == 32u) return rep_cut<32>(c);
            if (g == 16u) return rep_cut<16>(c);
            if (g == 8u) return rep_cut<8>(c);
            if (g == 4u) return rep_cut<4>(c);
            return p.force_direct ? exact_cut(c) : window_cut(c);
        }
    }

    // Every candidate of the row (at most k of them), in index order.
    __device__ void take_all(int32_t t0) {
        const int tid = threadIdx.x;
        stage_table(t0);
        uint32_t cnt = 0;
        for (int j = 0; j < NV; ++j) {
            uint32_t ck[4];
            clean(j * NT + tid, ck);
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) cnt += key_at<M>(ck, h) != 0u;
        }
        uint32_t total;
        uint32_t at = block_scan(s, par, cnt, total) - cnt;
        for (int j = 0; j < NV; ++j) {
            uint32_t ck[4];
            clean(j * NT + tid, ck);
#pragma unroll
            for (int h = 0; h < M::KPV; ++h)
                if (key_at<M>(ck, h) != 0u) put(at++, M::elem(j * NT + tid, h));
        }
        for (uint32_t i = total + threadIdx.x; i < k; i += NT)
            orow[i] = -1;
    }

    // The take lowest-index elements equal to c, written at out[first + rank].
    // Up to TIECAP of them are in s.tie_idx and ranked there; more are found
    // again in index order with scans of per-vector tie counts.
    __device__ void write_ties(uint32_t c, uint32_t take, uint32_t first, uint32_t e) {
        const uint32_t tid = threadIdx.x;
        if (e <= static_cast<uint32_t>(TIECAP)) {
            if (tid < e) {
                const uint32_t mine = s.tie_idx[tid];
                uint32_t r = tid;
                if (take < e) {
                    r = 0;
                    for (uint32_t u = 0; u < e; ++u) r += s.tie_idx[u] < mine;
                }
                if (r < take) put(first + r, mine);
            }
            return;
        }
        uint32_t before = 0;
        for (int j = 0; j < NV && before < take; ++j) {
            uint32_t ck[4];
            clean(j * NT + static_cast<int>(tid), ck);
            uint32_t eq = 0;
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) eq += key_at<M>(ck, h) == c;
            uint32_t total;
            uint32_t r = before + block_scan(s, par, eq, total) - eq;
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) {
                if (key_at<M>(ck, h) == c) {
                    if (r < take) put(first + r, M::elem(j * NT + static_cast<int>(tid), h));
                    ++r;
                }
            }
            before += total;
        }
    }

    // The q-th largest survivor when the window histogram cannot place it: a
    // two-pass radix select over s.surv_key[0 .. n), all in [lo, hi].
    __device__ uint32_t survivor_select(uint32_t n, uint32_t lo, uint32_t hi, uint32_t q, uint32_t &above) {
        const uint32_t tid = threadIdx.x;
        const uint32_t range = hi - lo;
        const int shift = range < 256u ? 0 : (32 - __clz(static_cast<int>(range))) - 8;
        const uint32_t mask = (1u << shift) - 1u;
        for (uint32_t i = tid; i < n; i += NT)
            atomicAdd(&s.hs[0][min((static_cast<uint32_t>(s.surv_key[i]) - lo) >> shift, 255u)], 1u);
        __syncthreads();
        warp0_find(s, s.hs[0], q);
        __syncthreads();
        const uint32_t b1 = s.bc[0], a1 = s.bc[1];
        __syncthreads();
        if (shift == 0) {
            above = a1;
            return lo + b1;
        }
        for (uint32_t i = tid; i < n; i += NT) {
            const uint32_t o = static_cast<uint32_t>(s.surv_key[i]) - lo;
            if ((o >> shift) == b1) atomicAdd(&s.hs[0][o & mask], 1u);
        }
        __syncthreads();
        warp0_find(s, s.hs[0], q - a1);
        __syncthreads();
        const uint32_t b2 = s.bc[0], a2 = s.bc[1];
        __syncthreads();
        above = a1 + a2;
        return lo + (b1 << shift) + b2;
    }

    // Survivors of cut c: every key >= c goes to the list, and to the window
    // histogram hw (bin key - c, the top bin holding every key >= c + 255).
    // Each thread tests its vectors' maxima; the vectors that may reach c are
    // queued per warp and worked through by all its lanes; slots come from one
    // warp scan and one shared atomic per round.
    template <bool FAST>
    __device__ __forceinline__ void survivors_t(uint32_t c, uint32_t *hw) {
        const uint32_t lane = lane_id(), warp = threadIdx.x >> 5, lt = (1u << lane) - 1u;
        const int32_t cs = static_cast<int32_t>(c) - 0x8000;
        uint32_t q = 0;
        bool pass[NV];  // every vector's test first: the loads issue together
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int pos = j * NT + static_cast<int>(threadIdx.x);
            if constexpr (FAST) pass[j] = pos < V && smax_halves(vec_smax(stg[pos])) >= cs;
            else if constexpr (M::BLOCK) pass[j] = bkey(pos) >= c;
            else pass[j] = pos < V && M::may_reach(stg[pos], 0u, c);
        }
        uint32_t bal[NV];  // every ballot first: the stores then only wait on popcounts
#pragma unroll
        for (int j = 0; j < NV; ++j) bal[j] = __ballot_sync(0xFFFFFFFFu, pass[j]);
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if (pass[j]) s.queue[warp][q + __popc(bal[j] & lt)] = static_cast<uint8_t>((j << 5) | lane);
            q += __popc(bal[j]);
        }
        __syncwarp();
        // Non-negative cut (FAST): the keys >= c are the BF16 bits >= c - 0x8000
        // as signed 16-bit integers, NaN excluded (its sign bit is set first).
        const uint32_t csm = (static_cast<uint32_t>(cs - 1) & 0xFFFFu) * 0x10001u;
        for (uint32_t e0 = 0; e0 < q; e0 += 32) {
            const uint32_t e = e0 + lane;
            uint32_t m = 0;
            int pos = 0;
            uint4 r = make_uint4(0, 0, 0, 0);
            uint32_t ck[4] = {0u, 0u, 0u, 0u};
            if (e < q) {
                const uint32_t qe = s.queue[warp][e];
                pos = static_cast<int>(qe >> 5) * NT + static_cast<int>(warp * 32u + (qe & 31u));
                if constexpr (FAST) {
                    // Bit i (i < 4): low half of word i; bit 4 + i: its high half.
                    r = stg[pos];
                    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
                    uint32_t u = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t x = w[i] | nan2(w[i]);
                        const uint32_t g = smax2(x, csm) ^ csm;  // nonzero halves: x >= cs
                        u |= ((((g & 0x7FFF7FFFu) + 0x7FFF7FFFu) | g) & 0x80008000u) >> (15 - i);
                    }
                    m = (u & 0xFu) | ((u >> 12) & 0xF0u);
                } else {
                    clean(pos, ck);
#pragma unroll
                    for (int h = 0; h < M::KPV; ++h) m |= (key_at<M>(ck, h) >= c ? 1u : 0u) << h;
                }
            }
            const uint32_t cnt = __popc(m);
            uint32_t tot;
            const uint32_t before = warp_excl_small(cnt, tot);
            uint32_t base = 0;
            if (lane == 0 && tot) base = atomicAdd(&s.v_cnt[rp], tot);
            uint32_t at = __shfl_sync(0xFFFFFFFFu, base, 0) + before;
#pragma unroll 1
            for (; m; m &= m - 1u) {
                const int bit = __ffs(m) - 1;
                uint32_t key, idx;
                if constexpr (FAST) {
                    const int i = bit & 3, hi = bit >> 2;
                    const uint32_t w = i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w;
                    key = ((hi ? w >> 16 : w) & 0xFFFFu) + 0x8000u;
                    idx = static_cast<uint32_t>(pos) * 8u + static_cast<uint32_t>(2 * i + hi);
                } else if constexpr (M::BLOCK) {
                    key = ck[0];
                    idx = static_cast<uint32_t>(pos);
                } else {
                    const int i = bit >> 1;
                    const uint32_t w = i == 0 ? ck[0] : i == 1 ? ck[1] : i == 2 ? ck[2] : ck[3];
                    key = (bit & 1) ? (w >> 16) : (w & 0xFFFFu);
                    idx = static_cast<uint32_t>(pos) * 8u + static_cast<uint32_t>(bit);
                }
                // Past the list's end (the count then exceeds it and the pass is
                // redone or replaced) writes go to the spare slot.
                const uint32_t slot = min(at, static_cast<uint32_t>(SURV_CAP));
                s.surv_key[slot] = static_cast<uint16_t>(key);
                s.surv_idx[slot] = idx;
                atomicAdd(&hw[min(key - c, 255u)], 1u);
                ++at;
            }
            __syncwarp();  // lanes left the loop above at different counts
        }
    }

    __device__ __forceinline__ void survivors(uint32_t c, uint32_t *hw) {
        if (!M::BLOCK && c >= 0x8000u) survivors_t<!M::BLOCK>(c, hw);
        else survivors_t<false>(c, hw);
    }

    // Warp 0: the bin b of window histogram h that holds the q-th largest key,
    // the count above it and the count in it, to s.bc; every bin from b up
    // becomes a cursor, the count of the bins above it (the output slot of its
    // first key). The caller's __syncthreads publishes both.
    __device__ __forceinline__ void warp0_cursors(uint32_t *h, uint32_t q) {
        if (threadIdx.x >= 32) return;
        __syncwarp();  // (see find_bin256)
        const uint32_t lane = lane_id();
        uint4 *h4 = reinterpret_cast<uint4 *>(h + 248 - 8 * static_cast<int>(lane));
        const uint4 a = h4[0], b = h4[1];
        const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) sum += v[i];
        const uint32_t incl = warp_incl_scan(sum);
        uint32_t acc = incl - sum, cur[8], bin = 0, above = 0, cnt = 0;
        bool mine = false;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
            cur[i] = acc;
            if (!mine && acc < q && acc + v[i] >= q) {
                mine = true;
                bin = 248u - 8u * lane + static_cast<uint32_t>(i);
                above = acc;
                cnt = v[i];
            }
            acc += v[i];
        }
        h4[0] = make_uint4(cur[0], cur[1], cur[2], cur[3]);
        h4[1] = make_uint4(cur[4], cur[5], cur[6], cur[7]);
        if (mine) {
            s.bc[0] = bin;
            s.bc[1] = above;
            s.bc[2] = cnt;
        }
        if (lane == 0) s.v_ntie = 0u;
    }

    // Output of the list against window h based at `base` (bins key - base)
    // whose bin b holds the k-th key: keys in higher bins take their bin's
    // next slot; keys in bin b too when every one of them is taken, otherwise
    // their indices go to s.tie_idx (while they fit) to be ranked.
    __device__ __forceinline__ void emit(uint32_t n, uint32_t *h, uint32_t base, uint32_t b, bool all_ties) {
        for (uint32_t i = threadIdx.x; i < n; i += NT) {
            const uint32_t key = s.surv_key[i];
            if (key < base) continue;
            const uint32_t bin = min(key - base, 255u);
            if (bin > b || (bin == b && all_ties)) {
                put(atomicAdd(&h[bin], 1u), s.surv_idx[i]);
            } else if (bin == b) {
                const uint32_t t = atomicAdd(&s.v_ntie, 1u);
                if (t < static_cast<uint32_t>(TIECAP)) s.tie_idx[t] = s.surv_idx[i];
            }
        }
    }

    // The exact cut c with more keys at or above it than the list holds (a
    // crowd of ties at c): keys > c in index order, then the lowest-index ties.
    __device__ void emit_rescan(uint32_t c) {
        const int tid = threadIdx.x;
        uint32_t before = 0;
        for (int j = 0; j < NV; ++j) {
            uint32_t ck[4];
            clean(j * NT + tid, ck);
            uint32_t gt = 0;
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) gt += key_at<M>(ck, h) > c;
            uint32_t total;
            uint32_t r = before + block_scan(s, par, gt, total) - gt;
#pragma unroll
            for (int h = 0; h < M::KPV; ++h)
                if (key_at<M>(ck, h) > c) put(r++, M::elem(j * NT + tid, h));
            before += total;
        }
        write_ties(c, k - before, before, 0xFFFFFFFFu);
    }

    // The cut for the next row: below the k-th key T by the distance that held
    // the n - k extra keys over [c, T], scaled to aim at about
    // k + min(max(k / 8, 128), (SURV_CAP - k) / 2) keys at or above it on a row
    // like this one. The margin covers the spread of the count, which grows like
    // its square root (measured on N(0,1) rows with k = 512: 128 left no row
    // short of k keys, 64 about one row in forty, each costing a second cut).
    __device__ __forceinline__ void next_guess(uint32_t c, uint32_t T, uint32_t n) {
        const uint32_t want = min(max(k / 8u, 128u), (static_cast<uint32_t>(SURV_CAP) - k) / 2u);
        const uint32_t d = T > c ? max((want * (T - c)) / (n - k + 1u), 1u) : 16u;
        guess = T > d ? T - d : 1u;
    }

    // Store the page ids loaded at the start of select() (the caller
    // synchronises before the first put).
    __device__ __forceinline__ void stage_table(int32_t t0) const {
        if (tab && threadIdx.x < static_cast<uint32_t>(TAB_CAP)) s.tab[threadIdx.x] = t0;
    }

    __device__ void select() {
        const uint32_t tid = threadIdx.x;
        const uint32_t nE = M::BLOCK ? static_cast<uint32_t>(V) : static_cast<uint32_t>(L);
        // The row's page ids, loaded now and staged in shared memory before the
        // first write (their latency hides behind the survivor pass).
        int32_t t0 = 0;  // page id of this thread's entry (TAB_CAP <= NT)
        tab = false;
        if (p.table) {
            const uint32_t npages = (nE + (1u << p.page_shift) - 1u) >> p.page_shift;
            if (npages <= static_cast<uint32_t>(TAB_CAP)) {
                tab = true;
                const int32_t *trow = table_row(p, row);
                if (tid < npages) t0 = __ldg(trow + tid);
            }
        }
        mask_tail();
        if (nE <= k) {
            count_event(p, TOPK_CNT_TILE_TAKE_ALL);
            take_all(t0);
            return;
        }
        // Group size: at least 2k representatives (and at least 4 logits).
        uint32_t g = 1;
        if (!p.force_direct) {
            // (groups are a thread's own vectors: at most NV blocks, 8 NV logits)
            if constexpr (M::BLOCK) {
                while (g < min(8u, static_cast<uint32_t>(NV)) && nE / (2u * g) >= 2u * k) g *= 2u;
            } else {
                g = 4;
                while (g < min(64u, 8u * NV) && nE / (2u * g) >= 2u * k) g *= 2u;
                if (nE / g < 2u * k) g = 1;  // too few groups of 4: exact path
            }
        }
        // First try the previous row's cut: any c with at least k keys >= c
        // bounds the k-th largest key from below, and the survivor pass counts
        // exactly those keys; a cut with too few of them or more than the list
        // holds is dropped for the representatives' cut.
        bool guessed = guess != 0u && !p.force_direct;
        // This row counts in s.v_cnt[rp] and s.hs[2 + rp], zeroed while the
        // previous row ran; the other pair, last used before the barrier that
        // ended the previous row, is zeroed now for the next one. A retry
        // zeroes its own pair, ordered before the new counts by the barriers of
        // the representatives' cut.
        rp ^= 1u;
        uint32_t *hw = s.hs[2 + rp];
        if (tid < 256u) s.hs[3 - rp][tid] = 0u;
        if (tid == 0) s.v_cnt[rp ^ 1u] = 0u;
        bool retry = false;
        for (;;) {
            PhaseClock clk;
            clk.start(p);
            if (retry) {
                if (tid < 256u) hw[tid] = 0u;
                if (tid == 0) s.v_cnt[rp] = 0u;
            }
            retry = true;
            uint32_t c = guess;
            if (!guessed && !cut_for(g, c)) {
                if (g > 1u) {  // the representatives cannot bound the row: exact path
                    count_event(p, TOPK_CNT_TILE_UNBOUNDED);
                    g = 1u;
                    __syncthreads();
                    continue;
                }
                count_event(p, TOPK_CNT_TILE_TAKE_ALL);
                take_all(t0);
                return;
            }
            clk.stop(p, TOPK_CNT_CYC_CUT);
            clk.start(p);
            survivors(c, hw);
            stage_table(t0);
            __syncthreads();
            clk.stop(p, TOPK_CNT_CYC_SURVIVORS);
            clk.start(p);
            const uint32_t n = s.v_cnt[rp];
            if (n < k || n > static_cast<uint32_t>(SURV_CAP)) {
                __syncthreads();
                if (guessed) {
                    count_event(p, TOPK_CNT_GUESS_MISS);
                    guessed = false;
                    continue;
                }
                if (n < k) {  // cannot happen: the cut is at most the k-th largest key
                    if (tid == 0) atomicOr(&g_device_status, ERR_BOUNDS);
                    return;
                }
                count_event(p, TOPK_CNT_TILE_OVERFLOW);
                if (g > 1u) {
                    g = 1u;
                    continue;
                }
                emit_rescan(c);  // the exact cut, with a crowd of ties at it
                guess = c > 16u ? c - 16u : 1u;
                clk.stop(p, TOPK_CNT_CYC_FINISH);
                return;
            }
            count_event(p, guessed ? TOPK_CNT_GUESS_HIT : g == 1u ? TOPK_CNT_TILE_EXACT : TOPK_CNT_TILE_SAMPLED);
            warp0_cursors(hw, k);
            __syncthreads();
            uint32_t b = s.bc[0], above = s.bc[1], e = s.bc[2];
            uint32_t T = c + b, base = c;
            uint32_t *h = hw;
            if (b == 255u) {
                // The k-th key is at least c + 255: find it by radix select over
                // the list, then emit against a window based at it.
                uint32_t smax = 0;
                for (uint32_t i = tid; i < n; i += NT) smax = max(smax, static_cast<uint32_t>(s.surv_key[i]));
                smax = __reduce_max_sync(0xFFFFFFFFu, smax);
                if (lane_id() == 0) atomicMax(&s.v_smax, smax);
                __syncthreads();
                uint32_t a2;
                T = survivor_select(n, c, s.v_smax, k, a2);
                if (tid == 0) s.v_smax = 0u;
                h = s.hs[1];
                base = T;
                for (uint32_t i = tid; i < n; i += NT) {
                    const uint32_t key = s.surv_key[i];
                    if (key >= T) atomicAdd(&h[min(key - T, 255u)], 1u);
                }
                __syncthreads();
                warp0_cursors(h, k);
                __syncthreads();
                b = s.bc[0];
                above = s.bc[1];
                e = s.bc[2];
            }
            clk.stop(p, TOPK_CNT_CYC_EXACT);
            clk.start(p);
            const uint32_t take = k - above;
            next_guess(c, T, n);
            emit(n, h, base, b, take == e);
            if (take != e) {
                __syncthreads();
                write_ties(T, take, above, e);
            }
            if (h != hw) {  // the cut's histogram back to zero
                __syncthreads();
                if (tid < 256u) h[tid] = 0u;
            }
            clk.stop(p, TOPK_CNT_CYC_FINISH);
            return;
        }
    }
};

static __device__ __forceinline__ void issue_row(Smem &s, int st, const Params &p, int32_t row, int32_t V) {
    const uint32_t bytes = static_cast<uint32_t>(V) * 16u;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.logits + static_cast<int64_t>(row) * p.row_stride);
    mbar_expect_tx(&s.full[st], bytes);
    bulk_load(&s.stage[st][0], src, bytes, &s.full[st]);
}

// The next row of this CTA, from `row` on in steps of `step`, that reads
// logits (p.rows when none is left); V = its valid vectors.
static __device__ __forceinline__ int32_t next_loaded_row(const Params &p, bool block, int32_t row, int32_t step,
                                                    int32_t &V) {
    for (; row < p.rows; row += step) {
        const int32_t L = min(max(__ldg(p.valid_len + row), 0), p.width);
        const int32_t n = block ? (L + 7) >> 3 : L;
        if (n > p.k) {
            V = (L + 7) >> 3;
            return row;
        }
    }
    return p.rows;
}

};  // struct Tile

template <class M, int NT, int SURV>
__global__ void __launch_bounds__(NT, NT == 256 ? (SURV <= 2048 ? 4 : 3) : 1) topk_one_tile_kernel(const Params p) {
    using O = Tile<NT, SURV>;
    constexpr int NSTAGE = O::NSTAGE;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    typename O::Smem &s = *reinterpret_cast<typename O::Smem *>(smem_raw);
    const int tid = threadIdx.x;
    const int32_t step = static_cast<int32_t>(gridDim.x);

    if (tid == 0) {  // (shared-memory set-up before the wait, as in topk_kernel)
        for (int i = 0; i < NSTAGE; ++i) mbar_init(&s.full[i], 1);
        fence_mbar_init();
        s.abort_flag = 0u;
        s.v_smax = 0u;
        s.v_cnt[0] = s.v_cnt[1] = 0u;
    }
    for (int i = tid; i < 4 * 256; i += NT) (&s.hs[0][0])[i] = 0u;
    __syncthreads();
    grid_dependency_wait();
    if (p.release) grid_dependents_release();

    int32_t feed_row = p.rows;
    if (tid == 0) {
        int32_t V;
        feed_row = O::next_loaded_row(p, M::BLOCK, static_cast<int32_t>(blockIdx.x), step, V);
        for (int i = 0; i < NSTAGE && feed_row < p.rows; ++i) {
            O::issue_row(s, i, p, feed_row, V);
            feed_row = O::next_loaded_row(p, M::BLOCK, feed_row + step, step, V);
        }
    }

    typename O::template Row<M> r(s, p);
    r.k = static_cast<uint32_t>(p.k);
    uint32_t seq = 0;
    for (int32_t row = static_cast<int32_t>(blockIdx.x); row < p.rows; row += step) {
        const int32_t L = min(max(__ldg(p.valid_len + row), 0), p.width);
        const int32_t n = M::BLOCK ? (L + 7) >> 3 : L;
        if (n <= p.k) {
            if (tid == 0) count_event(p, TOPK_CNT_BYPASS_ROWS);
            for (int32_t i = tid; i < p.k; i += NT)
                p.out[static_cast<int64_t>(row) * p.k + i] = i < n ? transform(p, row, i) : -1;
            continue;
        }
        const int st = static_cast<int>(seq & (NSTAGE - 1));
        r.row = row;
        r.L = L;
        r.V = (L + 7) >> 3;
        r.stg = s.stage[st];
        r.orow = p.out + static_cast<int64_t>(row) * p.k;
        PhaseClock clk;
        clk.start(p);
        mbar_wait(&s.full[st], (seq / NSTAGE) & 1u, &s.abort_flag);
        clk.stop(p, TOPK_CNT_CYC_WAIT);
        count_event(p, TOPK_CNT_ROUNDS);
        ++seq;
        clk.start(p);
        r.select();
        __syncthreads();  // every thread is done with this stage
        clk.stop(p, TOPK_CNT_CYC_SELECT);
        if (tid == 0 && feed_row < p.rows) {
            int32_t V;
            O::next_loaded_row(p, M::BLOCK, feed_row, step, V);
            fence_proxy_async();
            O::issue_row(s, st, p, feed_row, V);
            feed_row = O::next_loaded_row(p, M::BLOCK, feed_row + step, step, V);
        }
    }
}

}  // namespace one

// ------------------------------------------------------- ordered (tops) kernel
//
// The exact top-k of token rows in ascending index order, bounded by the
// scorer's per-8 maxima ("tops"): vLLM kimi_k3 "dsa/indexer", IndexerSelect
// (class docstring; write_selected). The k-th largest of a set of disjoint
// groups' maxima bounds the row's k-th key from below (each such group holds a
// key at least as large), so only the vectors whose top reaches that bound are
// read. One CTA of 512 threads per row:
//   1. representatives: maxima of groups of tops, each warp over its own
//      contiguous range of tops (coalesced 16-byte reads); the cut c is the
//      k-th largest representative, from a histogram of the 510 keys below the
//      largest one (two byte passes when it lies lower);
//   2. the vectors whose top is >= c, listed in index order (a second read of
//      the tops: counts, a CTA scan, then the writes);
//   3. every key >= c of those vectors, listed in index order (all threads load
//      their run of listed vectors together), binned by key - c;
//   4. the k-th key T from that histogram (or two byte passes over the list);
//   5. the output in index order: each listed key's slot is the number of
//      selected keys before it (keys above T, and ties at T while fewer than
//      the quota precede them), from one CTA scan.
// Rows whose lists would overflow, or whose representatives cannot bound the
// k-th key, take the exact select over every key (two radix passes, then the
// same ordered output from a scan of the row). Without tops every row does.
namespace ordered {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int REP_CAP = 16384;   // representatives: every top (rows of up to 16384 groups), else
                                 // every piece's maximum (up to 16384 pieces: 1M logits)
constexpr int VEC_CAP = 8192;    // candidate vectors listed
constexpr int KEY_CAP = 8192;    // candidate keys listed
constexpr int STAGE_VECS = (VEC_CAP * 4 + KEY_CAP * 6) / 16;  // rows the exact select keeps in shared memory
constexpr int MAX_BATCHES = 4;   // 256-piece batches of a warp's range of tops (16384 pieces / 16 warps)

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

struct alignas(16) Smem {
    alignas(16) uint32_t hs[2][256];  // byte-pass histograms (zero between uses)
    alignas(16) uint32_t hw[256];     // the candidates' window (key - c)
    uint16_t rep[REP_CAP];
    union {
        struct {
            uint32_t cvec[VEC_CAP];   // candidate vectors, in index order
            uint32_t lidx[KEY_CAP];   // candidate keys' element indices, in index order
            uint16_t lkey[KEY_CAP];
        };
        uint4 keys[STAGE_VECS];       // the exact select: a row's keys, 8 per vector (0: not eligible)
    };
    uint32_t red[2][NW];
    uint32_t bc[4];
    uint32_t plane[2048 / 32];        // B' words: bit 16 of each slot's index
};

__device__ __forceinline__ void count_o(const OParams &p, int which, uint32_t v = 1u) {
    if (p.counters && threadIdx.x == 0) atomicAdd(p.counters + which, v);
}

// The page transform of IndexerSelect.emit (request = row / q).
__device__ __forceinline__ int32_t transform_o(const OParams &p, int32_t row, int32_t i) {
    if (!p.table) return i;
    const int32_t request = p.rows_per_request == 1 ? row : row / p.rows_per_request;
    const int32_t page = p.table[static_cast<int64_t>(request) * p.table_stride + (i >> p.page_shift)];
    return page * p.block_rows + (i & ((1 << p.page_shift) - 1));
}

// Slot `slot` of the row's outputs: element i (transformed, and as is in ids);
// for B' words, (key << 16) | (0xFFFF - (i & 0xFFFF)) and bit 16 of i into the
// shared plane (written out with the row's last step).
__device__ __forceinline__ void put_o(const OParams &p, Smem &s, int32_t row, uint32_t slot, int32_t i,
                                      uint32_t key) {
    if (p.words) {
        p.out[static_cast<int64_t>(row) * (p.k + p.k / 32) + slot] =
            static_cast<int32_t>((key << 16) | (0xFFFFu - (static_cast<uint32_t>(i) & 0xFFFFu)));
        if ((i >> 16) & 1) atomicOr(&s.plane[slot >> 5], 1u << (slot & 31u));
        return;
    }
    const int64_t at = static_cast<int64_t>(row) * p.k + slot;
    p.out[at] = transform_o(p, row, i);
    if (p.ids) p.ids[at] = i;
}

// CTA-wide inclusive scan (every thread gets its prefix and the total).
__device__ __forceinline__ uint32_t cta_scan(Smem &s, uint32_t &par, uint32_t x, uint32_t &total) {
    const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
    const uint32_t inc = warp_incl_scan(x);
    if (lane == 31) s.red[par][warp] = inc;
    __syncthreads();
    const uint32_t w = lane < NW ? s.red[par][lane] : 0u;
    const uint32_t wi = warp_incl_scan(w);
    total = __shfl_sync(0xFFFFFFFFu, wi, 31);
    const uint32_t pre = __shfl_sync(0xFFFFFFFFu, wi - w, warp);
    par ^= 1u;
    return pre + inc;
}

// CTA-wide maximum.
__device__ __forceinline__ uint32_t cta_max(Smem &s, uint32_t &par, uint32_t x) {
    x = __reduce_max_sync(0xFFFFFFFFu, x);
    if (lane_id() == 0) s.red[par][threadIdx.x >> 5] = x;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < NW; ++w) x = max(x, s.red[par][w]);
    par ^= 1u;
    return x;
}

// Warp 0: the bin of hist holding the q-th largest, the count above it and
// the total, to s.bc; the histogram is zeroed. The caller's barrier publishes.
__device__ __forceinline__ void find_o(Smem &s, uint32_t *hist, uint32_t q) {
    if (threadIdx.x < 32) {
        uint32_t b, above, total;
        find_bin256(hist, q, b, above, total);
        reinterpret_cast<uint4 *>(hist)[2 * threadIdx.x] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4 *>(hist)[2 * threadIdx.x + 1] = make_uint4(0, 0, 0, 0);
        if (threadIdx.x == 0) {
            s.bc[0] = b;
            s.bc[1] = above;
            s.bc[2] = total;
        }
    }
}

// Bit h set when element h (0..7) of the vector has a key >= c (c >= 1);
// lanes at or past `len` elements of the row are not eligible, nor NaN.
__device__ __forceinline__ uint32_t mask_ge(const uint4 &r, uint32_t c, int32_t lanes) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t kk = key2(w[i]);
        const uint32_t lo = kk & 0xFFFFu, hi = kk >> 16;
        const bool nlo = ((w[i] & 0x7FFFu) > 0x7F80u), nhi = (((w[i] >> 16) & 0x7FFFu) > 0x7F80u);
        m |= (!nlo && lo >= c && 2 * i < lanes ? 1u : 0u) << (2 * i);
        m |= (!nhi && hi >= c && 2 * i + 1 < lanes ? 1u : 0u) << (2 * i + 1);
    }
    return m;
}

__device__ __forceinline__ uint32_t key_of8(const uint4 &r, int h) {
    const uint32_t w = (h & 4) ? ((h & 2) ? r.w : r.z) : ((h & 2) ? r.y : r.x);
    return (key2(w) >> ((h & 1) * 16)) & 0xFFFFu;
}

struct RowO {
    Smem &s;
    const OParams &p;
    uint32_t par = 0;
    int32_t row = 0, L = 0, V = 0;     // valid logits; vectors (and groups of tops) holding them
    uint32_t k = 0;
    const uint4 *lrow = nullptr;       // the row's logits as 16-byte vectors
    const uint4 *trow = nullptr;       // the row's tops, eight per 16 bytes

    __device__ RowO(Smem &s_, const OParams &p_) : s(s_), p(p_) {}

    __device__ __forceinline__ int32_t lanes_of(int32_t v) const { return min(8, L - 8 * v); }

    // Top g of the piece t (tops 8 * piece .. 8 * piece + 7); 0 past the row.
    __device__ __forceinline__ uint32_t top_at(const uint4 &t, int32_t piece, int e) const {
        const uint32_t w = (e & 4) ? ((e & 2) ? t.w : t.z) : ((e & 2) ? t.y : t.x);
        return 8 * piece + e < V ? (w >> ((e & 1) * 16)) & 0xFFFFu : 0u;
    }

    // Slots [from, k): -1 (words: 0); words also get the row's plane (the
    // caller's barrier has ordered every plane bit before this) and clear it.
    __device__ __forceinline__ void write_range_neg(uint32_t from) const {
        if (p.words) {
            int32_t *orow = p.out + static_cast<int64_t>(row) * (p.k + p.k / 32);
            for (uint32_t i = from + threadIdx.x; i < k; i += NT) orow[i] = 0;
            if (threadIdx.x < k / 32) {
                orow[k + threadIdx.x] = static_cast<int32_t>(s.plane[threadIdx.x]);
                s.plane[threadIdx.x] = 0u;
            }
            return;
        }
        for (uint32_t i = from + threadIdx.x; i < k; i += NT) {
            const int64_t at = static_cast<int64_t>(row) * p.k + i;
            p.out[at] = -1;
            if (p.ids) p.ids[at] = -1;
        }
    }

    // The k-th largest of the n representatives s.rep[0 .. n) (0 = none): a
    // window of the 510 keys at and below the largest, top (two keys per bin),
    // else two byte passes. The cut returned is at most it (the lower key of
    // the window bin that holds it); 0 when there are fewer than k
    // representatives.
    __device__ uint32_t rep_cut(uint32_t n, uint32_t top) {
        const uint32_t tid = threadIdx.x;
        const uint32_t slots = (n + NT - 1) / NT;
        for (uint32_t j = 0; j < slots; ++j) {
            const uint32_t i = j * NT + tid;
            const uint32_t v = i < n ? s.rep[i] : 0u;
            if (v) atomicAdd(&s.hw[255u - min((top - v) >> 1, 255u)], 1u);
        }
        __syncthreads();
        find_o(s, s.hw, k);
        __syncthreads();
        if (s.bc[2] < k) return 0u;
        const uint32_t b = s.bc[0];
        __syncthreads();  // every thread has read s.bc
        if (b > 0u) return static_cast<uint32_t>(max(static_cast<int>(top) - 2 * (255 - static_cast<int>(b)) - 1, 1));
        for (uint32_t j = 0; j < slots; ++j) {
            const uint32_t i = j * NT + tid;
            const uint32_t v = i < n ? s.rep[i] : 0u;
            agg_add(s.hs[0], v >> 8, v != 0u);
        }
        __syncthreads();
        find_o(s, s.hs[0], k);
        __syncthreads();
        const uint32_t hb = s.bc[0], ha = s.bc[1];
        __syncthreads();
        for (uint32_t j = 0; j < slots; ++j) {
            const uint32_t i = j * NT + tid;
            const uint32_t v = i < n ? s.rep[i] : 0u;
            const bool in = v != 0u && (v >> 8) == hb;
            if (__any_sync(0xFFFFFFFFu, in)) agg_add(s.hs[1], v & 0xFFu, in);
        }
        __syncthreads();
        find_o(s, s.hs[1], k - ha);
        __syncthreads();
        const uint32_t c = (hb << 8) | s.bc[0];
        __syncthreads();
        return c;
    }

    // The walk over the row's tops shared by steps 1 and 2: warp w takes the
    // pieces (8 tops, 16 bytes) [w * ppw, (w + 1) * ppw), in batches of 256,
    // lane l pieces p0 .. p0 + 7 of batch b, p0 = w * ppw + 256 b + 8 l (the
    // order of (b, l, u) is index order). Rows of at most REP_CAP groups keep
    // every top in s.rep (s.rep[g] = top g); longer ones every piece's maximum
    // (s.rep[piece]).
    struct Walk {
        int32_t pieces, ppw, base, end, batches;
        bool each;
    };
    __device__ __forceinline__ Walk walk() const {
        Walk w;
        w.pieces = (V + 7) / 8;
        w.ppw = (w.pieces + NW - 1) / NW;
        w.base = static_cast<int32_t>(threadIdx.x >> 5) * w.ppw;
        w.end = min(w.base + w.ppw, w.pieces);
        w.batches = (w.ppw + 255) / 256;
        w.each = V <= REP_CAP;
        return w;
    }

    // Step 1: the cut from the tops (0: none).
    __device__ uint32_t cut_from_tops() {
        const Walk w = walk();
        if (w.batches > MAX_BATCHES) {  // (rows are at most 1M logits: cannot happen)
            if (threadIdx.x == 0) atomicOr(&g_device_status, ERR_BOUNDS);
            return 0u;
        }
        // Read coalesced: at round j lane l takes pieces base + 256 j + 32 u + l,
        // u < 8 (the eight loads issue together); kept by piece index.
        uint32_t best = 0;
        for (int32_t b = 0; b < w.batches; ++b) {
            uint4 t[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int32_t pc = w.base + 256 * b + 32 * u + static_cast<int32_t>(lane_id());
                t[u] = pc < w.end ? __ldg(trow + pc) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int32_t pc = w.base + 256 * b + 32 * u + static_cast<int32_t>(lane_id());
                if (pc >= w.end) continue;
                uint32_t acc = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t top = top_at(t[u], pc, e);
                    if (w.each) s.rep[8 * pc + e] = static_cast<uint16_t>(top);
                    acc = max(acc, top);
                }
                if (!w.each) s.rep[pc] = static_cast<uint16_t>(acc);
                best = max(best, acc);
            }
        }
        const uint32_t top = cta_max(s, par, best);  // (its barrier also publishes s.rep)
        if (top == 0u) return 0u;  // no eligible key at all
        return rep_cut(static_cast<uint32_t>(w.each ? 8 * w.pieces : w.pieces), top);
    }

    // Step 2: the vectors whose top is >= c, in index order, into s.cvec: from
    // the tops kept in s.rep, or, for long rows, from the pieces whose maximum
    // in s.rep reaches c (only those are read again). A counting pass, the
    // warps' offsets, then the writes. Returns the count (listed only up to
    // VEC_CAP).
    __device__ uint32_t list_vectors(uint32_t c) {
        const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
        const Walk w = walk();
        uint64_t mk[MAX_BATCHES];  // bit 8u + e: top e of the lane's piece u of batch b is >= c
        uint32_t cnt = 0;
        if (w.each) {
#pragma unroll
            for (int b = 0; b < MAX_BATCHES; ++b) {
                mk[b] = 0;
                if (b >= w.batches) continue;
                const int32_t p0 = w.base + 256 * b + 8 * static_cast<int32_t>(lane);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (p0 + u >= w.end) continue;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        mk[b] |= static_cast<uint64_t>(s.rep[8 * (p0 + u) + e] >= c ? 1u : 0u) << (8 * u + e);
                }
                cnt += __popcll(mk[b]);
            }
        } else {
            // Pieces whose maximum reaches c (bit 8b + u), then their tops, read
            // four at a time with the loads issued together.
            uint32_t flags = 0;
#pragma unroll
            for (int b = 0; b < MAX_BATCHES; ++b) {
                mk[b] = 0;
                const int32_t p0 = w.base + 256 * b + 8 * static_cast<int32_t>(lane);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (b < w.batches && p0 + u < w.end && s.rep[p0 + u] >= c) flags |= 1u << (8 * b + u);
            }
            while (flags) {
                int f[4];
                uint4 t[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    f[x] = flags ? __ffs(flags) - 1 : -1;
                    if (flags) flags &= flags - 1u;
                    const int32_t pc = w.base + 256 * (f[x] >> 3) + 8 * static_cast<int32_t>(lane) + (f[x] & 7);
                    t[x] = f[x] >= 0 ? __ldg(trow + pc) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    if (f[x] < 0) continue;
                    const int32_t pc = w.base + 256 * (f[x] >> 3) + 8 * static_cast<int32_t>(lane) + (f[x] & 7);
                    uint64_t m = 0;
#pragma unroll
                    for (int e = 0; e < 8; ++e) m |= static_cast<uint64_t>(top_at(t[x], pc, e) >= c ? 1u : 0u) << e;
#pragma unroll
                    for (int b = 0; b < MAX_BATCHES; ++b)
                        if ((f[x] >> 3) == b) mk[b] |= m << (8 * (f[x] & 7));
                }
            }
#pragma unroll
            for (int b = 0; b < MAX_BATCHES; ++b) cnt += __popcll(mk[b]);
        }
        const uint32_t wt = __reduce_add_sync(0xFFFFFFFFu, cnt);
        if (lane == 0) s.red[par][warp] = wt;
        __syncthreads();
        uint32_t at = 0, total = 0;
        for (uint32_t x = 0; x < static_cast<uint32_t>(NW); ++x) {
            const uint32_t y = s.red[par][x];
            at += x < warp ? y : 0u;
            total += y;
        }
        par ^= 1u;
        if (total > static_cast<uint32_t>(VEC_CAP)) return total;
#pragma unroll
        for (int b = 0; b < MAX_BATCHES; ++b) {
            if (b >= w.batches) break;  // (uniform)
            uint64_t m = mk[b];
            const uint32_t n = __popcll(m);
            const uint32_t incl = warp_incl_scan(n);
            uint32_t pos = at + incl - n;
            const int32_t p0 = w.base + 256 * b + 8 * static_cast<int32_t>(lane);
            for (; m; m &= m - 1u) s.cvec[pos++] = static_cast<uint32_t>(8 * p0 + __ffsll(m) - 1);
            at += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        __syncthreads();
        return total;
    }

    // Step 3: every key >= c of the nv listed vectors, in index order, into
    // s.lkey / s.lidx, binned by key - c into s.hw (the last bin open-ended).
    // Thread t takes listed vectors [t q, t q + q). Returns the count (listed
    // only up to KEY_CAP).
    __device__ uint32_t list_keys(uint32_t c, uint32_t nv) {
        constexpr uint32_t HOLD = 8;  // vectors a thread keeps in registers between the passes
        const uint32_t tid = threadIdx.x;
        const uint32_t q = (nv + NT - 1) / NT;
        const uint32_t j0 = min(tid * q, nv), j1 = min(j0 + q, nv);
        uint4 r[HOLD];
#pragma unroll
        for (uint32_t u = 0; u < HOLD; ++u)  // the loads issue together
            r[u] = j0 + u < j1 ? __ldg(lrow + s.cvec[j0 + u]) : make_uint4(0u, 0u, 0u, 0u);
        uint32_t cnt = 0;
#pragma unroll
        for (uint32_t u = 0; u < HOLD; ++u)
            if (j0 + u < j1) cnt += __popc(mask_ge(r[u], c, lanes_of(static_cast<int32_t>(s.cvec[j0 + u]))));
        for (uint32_t j = j0 + HOLD; j < j1; ++j) {  // runs longer than HOLD (few rows)
            const uint4 x = __ldg(lrow + s.cvec[j]);
            cnt += __popc(mask_ge(x, c, lanes_of(static_cast<int32_t>(s.cvec[j]))));
        }
        uint32_t total;
        uint32_t at = cta_scan(s, par, cnt, total) - cnt;
        if (total > static_cast<uint32_t>(KEY_CAP)) return total;
        auto put_keys = [&](const uint4 &x, int32_t v) {
            for (uint32_t m = mask_ge(x, c, lanes_of(v)); m; m &= m - 1u) {
                const int h = __ffs(m) - 1;
                const uint32_t key = key_of8(x, h);
                s.lkey[at] = static_cast<uint16_t>(key);
                s.lidx[at] = static_cast<uint32_t>(8 * v + h);
                atomicAdd(&s.hw[min(key - c, 255u)], 1u);
                ++at;
            }
        };
#pragma unroll
        for (uint32_t u = 0; u < HOLD; ++u)
            if (j0 + u < j1) put_keys(r[u], static_cast<int32_t>(s.cvec[j0 + u]));
        for (uint32_t j = j0 + HOLD; j < j1; ++j) put_keys(__ldg(lrow + s.cvec[j]), static_cast<int32_t>(s.cvec[j]));
        __syncthreads();
        return total;
    }

    // Step 5 (and the exact path's output): n_own entries of this thread, in
    // index order, after those of lower threads; slot of each selected one =
    // the selected entries before it in index order (keys above T, then ties
    // at T while fewer than `take` precede them).
    template <class Get>
    __device__ __forceinline__ void write_ordered(uint32_t T, uint32_t take, bool all, uint32_t n_own, Get &&get) {
        uint32_t gt = 0, eq = 0;
        for (uint32_t j = 0; j < n_own; ++j) {
            uint32_t key;
            int32_t idx;
            get(j, key, idx);
            gt += key > T || (all && key != 0u);
            eq += !all && key == T && key != 0u;
        }
        uint32_t tg, te;
        uint32_t pa = cta_scan(s, par, gt, tg) - gt;
        uint32_t pt = cta_scan(s, par, eq, te) - eq;
        if (gt == 0u && (eq == 0u || pt >= take)) return;
        for (uint32_t j = 0; j < n_own; ++j) {
            uint32_t key;
            int32_t idx;
            get(j, key, idx);
            if (key == 0u) continue;
            // Ordered: the selected keys before it in index order. Words:
            // the keys above in index order, then the ties taken.
            if (key > T || all) {
                put_o(p, s, row, p.words ? pa : pa + min(pt, take), idx, key);
                ++pa;
            } else if (key == T) {
                if (pt < take) put_o(p, s, row, p.words ? k - take + pt : pa + pt, idx, key);
                ++pt;
            }
        }
    }

    // The keys of vector v (element h in half h of the result; 0: not eligible).
    __device__ __forceinline__ uint4 packed_keys(int32_t v) const {
        const uint4 r = __ldg(lrow + v);
        const uint32_t m = mask_ge(r, 1u, lanes_of(v));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t kk = key2(w[i]);
            o[i] = (((m >> (2 * i)) & 1u) ? kk & 0xFFFFu : 0u) | (((m >> (2 * i + 1)) & 1u) ? kk & 0xFFFF0000u : 0u);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }

    static __device__ __forceinline__ uint32_t half8(const uint4 &kk, int h) {
        const uint32_t w = (h & 4) ? ((h & 2) ? kk.w : kk.z) : ((h & 2) ? kk.y : kk.x);
        return (w >> ((h & 1) * 16)) & 0xFFFFu;
    }

    // The exact select over every key of the row, then the ordered output from
    // a scan of the row: thread t takes vectors [t q, t q + q). The k-th key:
    // the row's largest key M and the eligible count (one pass), a histogram of
    // the 512 keys below M in bins of two (the keys in it spread over the bins:
    // plain atomics), then which of the bin's two keys it is (a count of the
    // upper one); when it lies lower, two byte passes over every key. Rows of at
    // most STAGE_VECS vectors keep their keys in shared memory after the first
    // pass (the lists are not in use).
    __device__ void exact_row() {
        const uint32_t tid = threadIdx.x;
        count_o(p, TOPK_CNT_ORDERED_EXACT);
        const bool staged = V <= STAGE_VECS;
        auto keys_of = [&](int32_t v) -> uint4 { return staged ? s.keys[v] : packed_keys(v); };
        uint32_t top = 0, mine = 0;
        for (int32_t v0 = 0; v0 < V; v0 += NT) {
            const int32_t v = v0 + static_cast<int32_t>(tid);
            const uint4 kk = v < V ? packed_keys(v) : make_uint4(0u, 0u, 0u, 0u);
            if (staged && v < V) s.keys[v] = kk;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const uint32_t key = half8(kk, h);
                top = max(top, key);
                mine += key != 0u;
            }
        }
        uint32_t total;
        cta_scan(s, par, mine, total);  // (its barrier also publishes the staged keys)
        top = cta_max(s, par, top);
        uint32_t T = 0, take = 0;
        const bool all = total <= k;  // every eligible key
        bool found = all;
        if (!all) {
            const uint32_t lo = top > 511u ? top - 511u : 1u;  // the window: keys lo .. top
            for (int32_t v0 = 0; v0 < V; v0 += NT) {
                const int32_t v = v0 + static_cast<int32_t>(tid);
                const uint4 kk = v < V ? keys_of(v) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const uint32_t key = half8(kk, h);
                    if (key >= lo) atomicAdd(&s.hs[0][255u - ((top - key) >> 1)], 1u);
                }
            }
            __syncthreads();
            find_o(s, s.hs[0], k);
            __syncthreads();
            const uint32_t b = s.bc[0], above_b = s.bc[1], in_window = s.bc[2];
            __syncthreads();
            if (in_window >= k) {
                // Bin b holds keys top - 2 (255 - b) - 1 and the one above it.
                const uint32_t upper = top - 2u * (255u - b);
                uint32_t n_up = 0;
                for (int32_t v0 = 0; v0 < V; v0 += NT) {
                    const int32_t v = v0 + static_cast<int32_t>(tid);
                    const uint4 kk = v < V ? keys_of(v) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int h = 0; h < 8; ++h) n_up += half8(kk, h) == upper;
                }
                uint32_t ups;
                cta_scan(s, par, n_up, ups);
                if (above_b + ups >= k) {
                    T = upper;
                    take = k - above_b;
                } else {
                    T = upper - 1u;
                    take = k - above_b - ups;
                }
                found = true;
            }
        }
        if (!found) {
            for (int32_t v0 = 0; v0 < V; v0 += NT) {
                const int32_t v = v0 + static_cast<int32_t>(tid);
                const uint4 kk = v < V ? keys_of(v) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const uint32_t key = half8(kk, h);
                    agg_add(s.hs[0], key >> 8, key != 0u);
                }
            }
            __syncthreads();
            find_o(s, s.hs[0], k);
            __syncthreads();
            const uint32_t hb = s.bc[0], ha = s.bc[1];
            __syncthreads();
            for (int32_t v0 = 0; v0 < V; v0 += NT) {
                const int32_t v = v0 + static_cast<int32_t>(tid);
                const uint4 kk = v < V ? keys_of(v) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const uint32_t key = half8(kk, h);
                    const bool in = key != 0u && (key >> 8) == hb;
                    if (__any_sync(0xFFFFFFFFu, in)) agg_add(s.hs[1], key & 0xFFu, in);
                }
            }
            __syncthreads();
            find_o(s, s.hs[1], k - ha);
            __syncthreads();
            T = (hb << 8) | s.bc[0];
            take = k - ha - s.bc[1];
            __syncthreads();
        }
        const uint32_t q = (static_cast<uint32_t>(V) + NT - 1) / NT;
        const uint32_t v0 = min(tid * q, static_cast<uint32_t>(V)), v1 = min(v0 + q, static_cast<uint32_t>(V));
        uint32_t gt = 0, eq = 0;
        for (uint32_t v = v0; v < v1; ++v) {
            const uint4 kk = keys_of(static_cast<int32_t>(v));
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const uint32_t key = half8(kk, h);
                gt += key != 0u && (key > T || all);
                eq += !all && key != 0u && key == T;
            }
        }
        uint32_t tg, te;
        uint32_t pa = cta_scan(s, par, gt, tg) - gt;
        uint32_t pt = cta_scan(s, par, eq, te) - eq;
        if (gt != 0u || (eq != 0u && pt < take)) {
            for (uint32_t v = v0; v < v1; ++v) {
                const uint4 kk = keys_of(static_cast<int32_t>(v));
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const uint32_t key = half8(kk, h);
                    if (key == 0u) continue;
                    const int32_t idx = static_cast<int32_t>(8 * v) + h;
                    if (key > T || all) {
                        put_o(p, s, row, p.words ? pa : pa + min(pt, take), idx, key);
                        ++pa;
                    } else if (key == T) {
                        if (pt < take) put_o(p, s, row, p.words ? k - take + pt : pa + pt, idx, key);
                        ++pt;
                    }
                }
            }
        }
        const uint32_t selected = all ? total : k;
        if (p.words) __syncthreads();  // every plane bit set
        write_range_neg(selected);
        if (tid == 0) p.valid[row] = static_cast<int32_t>(selected);
    }

    __device__ void select(int32_t row_) {
        const uint32_t tid = threadIdx.x;
        row = row_;
        k = static_cast<uint32_t>(p.k);
        L = min(max(__ldg(p.valid_len + row), 0), p.width);
        V = (L + 7) / 8;
        lrow = reinterpret_cast<const uint4 *>(p.logits + static_cast<int64_t>(row) * p.row_stride);
        if (p.words && static_cast<uint32_t>(L) <= k) {  // the whole row, its keys in the words
            count_o(p, TOPK_CNT_BYPASS_ROWS);
            const uint16_t *x = p.logits + static_cast<int64_t>(row) * p.row_stride;
            int32_t *orow = p.out + static_cast<int64_t>(row) * (p.k + p.k / 32);
            for (uint32_t j = tid; j < k; j += NT) {
                uint32_t w = 0;
                if (j < static_cast<uint32_t>(L)) {
                    const uint32_t b = x[j];
                    w = ((b ^ ((b & 0x8000u) ? 0xFFFFu : 0x8000u)) << 16) | (0xFFFFu - (j & 0xFFFFu));
                }
                orow[j] = static_cast<int32_t>(w);
            }
            for (uint32_t t = tid; t < k / 32; t += NT) {  // bit 16 of the indices 32 t .. 32 t + 31 below L
                uint32_t m = 0;
                for (uint32_t b = 0; b < 32; ++b) {
                    const uint32_t j = 32 * t + b;
                    m |= (j < static_cast<uint32_t>(L) && ((j >> 16) & 1u)) ? 1u << b : 0u;
                }
                orow[k + t] = static_cast<int32_t>(m);
            }
            if (tid == 0) p.valid[row] = L;
            return;
        }
        if (static_cast<uint32_t>(L) <= k) {  // the whole row, values not read
            count_o(p, TOPK_CNT_BYPASS_ROWS);
            for (uint32_t i = tid; i < k; i += NT) {
                const int64_t at = static_cast<int64_t>(row) * p.k + i;
                p.out[at] = i < static_cast<uint32_t>(L) ? transform_o(p, row, static_cast<int32_t>(i)) : -1;
                if (p.ids) p.ids[at] = i < static_cast<uint32_t>(L) ? static_cast<int32_t>(i) : -1;
            }
            if (tid == 0) p.valid[row] = L;
            return;
        }
        if (!p.tops) {
            exact_row();
            return;
        }
        trow = reinterpret_cast<const uint4 *>(p.tops + static_cast<int64_t>(row) * p.tops_stride);
        const uint32_t c = cut_from_tops();
        if (c == 0u) {
            exact_row();
            return;
        }
        const uint32_t nv = list_vectors(c);
        if (nv > static_cast<uint32_t>(VEC_CAP)) {
            exact_row();
            return;
        }
        const uint32_t nk = list_keys(c, nv);
        if (nk > static_cast<uint32_t>(KEY_CAP) || nk < k) {  // (nk < k: tops not the row's maxima)
            if (nk < k && tid == 0) atomicOr(&g_device_status, ERR_BOUNDS);
            if (tid < 256u) s.hw[tid] = 0u;
            __syncthreads();
            exact_row();
            return;
        }
        count_o(p, TOPK_CNT_ORDERED_TOPS);
        // Step 4: the k-th key T.
        find_o(s, s.hw, k);
        __syncthreads();
        uint32_t b = s.bc[0], above = s.bc[1];
        __syncthreads();
        uint32_t T = c + b;
        if (b == 255u) {  // at least c + 255: two byte passes over key - c of the list
            for (uint32_t i0 = 0; i0 < nk; i0 += NT) {
                const uint32_t i = i0 + tid;
                const uint32_t d = i < nk ? static_cast<uint32_t>(s.lkey[i]) - c : 0u;
                agg_add(s.hs[0], d >> 8, i < nk);
            }
            __syncthreads();
            find_o(s, s.hs[0], k);
            __syncthreads();
            const uint32_t hb = s.bc[0], ha = s.bc[1];
            __syncthreads();
            for (uint32_t i0 = 0; i0 < nk; i0 += NT) {
                const uint32_t i = i0 + tid;
                const uint32_t d = i < nk ? static_cast<uint32_t>(s.lkey[i]) - c : 0u;
                const bool in = i < nk && (d >> 8) == hb;
                if (__any_sync(0xFFFFFFFFu, in)) agg_add(s.hs[1], d & 0xFFu, in);
            }
            __syncthreads();
            find_o(s, s.hs[1], k - ha);
            __syncthreads();
            T = c + ((hb << 8) | s.bc[0]);
            above = ha + s.bc[1];
            __syncthreads();
        }
        // Step 5: the ordered output; thread t takes list entries [t q, t q + q).
        const uint32_t q = (nk + NT - 1) / NT;
        const uint32_t i0 = min(tid * q, nk), i1 = min(i0 + q, nk);
        write_ordered(T, k - above, false, i1 - i0, [&](uint32_t j, uint32_t &key, int32_t &idx) {
            key = s.lkey[i0 + j];
            idx = static_cast<int32_t>(s.lidx[i0 + j]);
        });
        if (p.words) {
            __syncthreads();  // every plane bit set
            write_range_neg(k);
        }
        if (tid == 0) p.valid[row] = static_cast<int32_t>(k);
    }
};

__global__ void __launch_bounds__(NT, 1) topk_ordered_kernel(const OParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Smem &s = *reinterpret_cast<Smem *>(smem_raw);
    if (threadIdx.x < 256u) s.hs[0][threadIdx.x] = s.hs[1][threadIdx.x] = s.hw[threadIdx.x] = 0u;
    if (threadIdx.x < 2048u / 32u) s.plane[threadIdx.x] = 0u;
    __syncthreads();
    grid_dependency_wait();
    if (p.release) grid_dependents_release();

    RowO r(s, p);
    for (int32_t row = static_cast<int32_t>(blockIdx.x); row < p.rows; row += static_cast<int32_t>(gridDim.x)) {
        r.select(row);
        __syncthreads();
    }
}

// The per-8 maxima: thread i of the grid takes piece i (8 groups of 8 logits)
// of its row and writes their tops as one 16-byte store. A group's top is the
// largest key among its logits below the row's valid length that are not NaN,
// 0 when there is none.
__global__ void __launch_bounds__(256) topk_tops_kernel(const uint16_t *logits, int64_t row_stride,
                                                        int32_t rows, int32_t width,
                                                        const int32_t *valid_len, uint16_t *tops,
                                                        int64_t tops_stride, int32_t pieces) {
    grid_dependency_wait();
    grid_dependents_release();
    const int64_t total = static_cast<int64_t>(rows) * pieces;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t row = static_cast<int32_t>(i / pieces), piece = static_cast<int32_t>(i % pieces);
        const int32_t L = min(max(__ldg(valid_len + row), 0), width);
        const uint4 *src = reinterpret_cast<const uint4 *>(logits + static_cast<int64_t>(row) * row_stride);
        uint32_t t[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int32_t v = 8 * piece + e;
            uint32_t top = 0;
            if (8 * v < L) {
                const uint4 r = __ldg(src + v);
                const uint32_t m = mask_ge(r, 1u, min(8, L - 8 * v));
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    if ((m >> h) & 1u) top = max(top, key_of8(r, h));
            }
            t[e] = top;
        }
        reinterpret_cast<uint4 *>(tops + static_cast<int64_t>(row) * tops_stride)[piece] =
            make_uint4(t[0] | (t[1] << 16), t[2] | (t[3] << 16), t[4] | (t[5] << 16), t[6] | (t[7] << 16));
    }
}

}  // namespace ordered

// ------------------------------------------------------------------ host side

struct Variant {
    const void *fn;
    int smem;
};

constexpr int WIDE_NSTAGE = 2, WIDE_CAP = 4096;

template <class M, int NSTAGE, int CAP>
Variant variant() {
    return Variant{reinterpret_cast<const void *>(&topk_kernel<M, NSTAGE, CAP>),
                   static_cast<int>(sizeof(Smem<NSTAGE, CAP>))};
}

template <class M, int NT, int SURV>
Variant one_variant() {
    return Variant{reinterpret_cast<const void *>(&one::topk_one_tile_kernel<M, NT, SURV>),
                   static_cast<int>(sizeof(typename one::Tile<NT, SURV>::Smem))};
}

// build 0: 256 threads, k <= 1024; 1: 256 threads, larger k; 2: 512 threads
// (rows that do not fill the SMs).
constexpr int ONE_BUILDS = 3;
Variant pick_one(bool block, int build) {
    switch (build) {
        case 0: return block ? one_variant<BlockMode, 256, 2048>() : one_variant<TokenMode, 256, 2048>();
        case 1: return block ? one_variant<BlockMode, 256, 4096>() : one_variant<TokenMode, 256, 4096>();
        default: return block ? one_variant<BlockMode, 512, 4096>() : one_variant<TokenMode, 512, 4096>();
    }
}

// The streamed kernel (rows wider than one tile, or split over a cluster).
Variant pick(bool block, bool) {
    return block ? variant<BlockMode, WIDE_NSTAGE, WIDE_CAP>() : variant<TokenMode, WIDE_NSTAGE, WIDE_CAP>();
}

// The resident-keys kernel (block rows wider than one tile).
Variant pick_direct(bool block) {
    return block ? Variant{reinterpret_cast<const void *>(&direct::topk_direct_kernel<BlockMode>),
                           static_cast<int>(sizeof(direct::Smem))}
                 : Variant{reinterpret_cast<const void *>(&direct::topk_direct_kernel<TokenMode>),
                           static_cast<int>(sizeof(direct::Smem))};
}

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
                const Variant v = pick(b != 0, true);
                e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem);
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e == cudaSuccess)
                    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.per_sm[b][w], v.fn, THREADS,
                                                                      static_cast<size_t>(v.smem));
                if (e == cudaSuccess && d.per_sm[b][w] < 1) e = cudaErrorInvalidConfiguration;
            }
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            const Variant v = pick_direct(b != 0);
            e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.per_sm_direct[b], v.fn, direct::NT,
                                                                  static_cast<size_t>(v.smem));
            if (e == cudaSuccess && d.per_sm_direct[b] < 1) e = cudaErrorInvalidConfiguration;
        }
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(reinterpret_cast<const void *>(&ordered::topk_ordered_kernel),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(sizeof(ordered::Smem)));
        for (int b = 0; b < 2 && e == cudaSuccess; ++b)
            for (int l = 0; l < 5; ++l) {
                const int c = 1 << l;
                d.cap[0][b][l] = l == 0 ? d.sms * d.per_sm[b][1] : cluster_capacity(pick(b != 0, true), THREADS, c);
                d.cap[1][b][l] = l == 0 ? d.sms * d.per_sm_direct[b]
                                        : cluster_capacity(pick_direct(b != 0), direct::NT, c);
            }
        for (int b = 0; b < 2 && e == cudaSuccess; ++b)
            for (int w = 0; w < ONE_BUILDS && e == cudaSuccess; ++w) {
                const Variant v = pick_one(b != 0, w);
                e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem);
                if (e == cudaSuccess)
                    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.per_sm_one[b][w], v.fn, w == 2 ? 512 : 256,
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
    int build;         // one-tile rows: which build (see pick_one)
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
        pl.threads = pl.build == 2 ? 512 : 256;
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
    const Variant v = pl.kind == KIND_ONE ? pick_one(block, pl.build)
                      : pl.kind == KIND_STREAM ? pick(block, true) : pick_direct(block);
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
    cfg.dynamicSmemBytes = sizeof(ordered::Smem);
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
    const cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(&ordered::topk_ordered_kernel), args);
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
    topk::ordered::topk_tops_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        logits, row_stride, rows, width, valid_len, tops, tops_stride, static_cast<int32_t>(pieces));
    return cudaGetLastError() == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
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
    const topk::Variant v = pl.kind == topk::KIND_ONE ? topk::pick_one(block, pl.build)
                            : pl.kind == topk::KIND_STREAM ? topk::pick(block, true) : topk::pick_direct(block);
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
    if (cudaMemcpyFromSymbol(&v, topk::g_device_status, sizeof(v)) != cudaSuccess) return TOPK_ERR_CUDA;
    if (flags) *flags = v;
    if (clear) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(topk::g_device_status, &zero, sizeof(zero)) != cudaSuccess)
            return TOPK_ERR_CUDA;
    }
    return TOPK_OK;
}

}  // extern "C"
