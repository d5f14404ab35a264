// Exact per-row top-k of BF16 logits for GB300 (sm_103a): the streamed cluster
// kernel, for token rows wider than one 32 KiB stage.
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
// selected exactly. Its cutoff comes from group representatives: one element
// of each group (token rows with room for 2k of them: every 16-byte vector, its
// largest logit, held in registers; otherwise groups of 4 to 64 elements). The
// k-th largest representative bounds the tile's k-th key from below, because k
// distinct elements reach it; keys above it sit in about k groups, so they are
// few. Those survivors go to the buffer and their exact k-th comes from a
// histogram relative to the cutoff. When the representatives cannot bound the
// tile, or the survivors overflow, every key becomes its own representative
// (g = 1): the exact path. Later tiles append every key at or above a running
// threshold, which rises whenever the buffer is compacted to its top-k and, in
// a cluster, when a peer CTA publishes its own bound through distributed shared
// memory. A launch whose clusters take one row each may instead start every
// row at the threshold its cluster slot carried over from the previous launch
// (see g_stream_carry), checked on the first tiles and by the final counts.
//
// In token rows every thread forms the 8-bit masks of its vectors' logits at
// or above the threshold with packed BF16 compares (NaN never passes), and a
// warp reserves the slots of all its survivors with one shared atomic, never
// one per key; block rows queue the candidate vectors per warp (ballots) and
// the warp's lanes work through the queue together. The C buffers
// of a row are merged with cluster-wide histograms over distributed shared
// memory; ties at the row's k-th key are split across CTAs in index order, and
// each CTA writes its part of the answer through the block table, every
// output slot from one CTA scan of (ties, above) counts.
// The packed BF16 compares decide exactly what a compare of the 16-bit keys
// decides (NaN never passes); every count, cut and histogram is on the keys.

#include "common.cuh"

namespace topk {

// Carried thresholds: each cluster slot keeps the k-th key of the last row it
// selected (tagged with the mode and k). A launch whose clusters take at most
// one row each starts every row at that key less STREAM_CARRY_MARGIN, which
// the row's own buffers then accept (k keys at or above it) or reject (the row
// is streamed again without it): a starting point only. A word whose row
// dropped its threshold carries STREAM_CARRY_DROPPED: the next launch does not
// try it (rows whose distribution changes from launch to launch then pay the
// first-tile check every other launch only).
constexpr int STREAM_CARRY_SLOTS = 512;
constexpr uint32_t STREAM_CARRY_MARGIN = 16;
constexpr uint32_t STREAM_CARRY_DROPPED = 1u << 30;
constexpr uint32_t STREAM_CARRY_TAG_MASK = 0x8FFF0000u;  // mode (bit 31) and k (bits 16-27)
static __device__ uint32_t g_stream_carry[STREAM_CARRY_SLOTS];

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
    uint32_t carry_word;                     // rank 0: the carried word this launch starts from
    uint32_t guess_cnt, guess_nv;            // rank 0: keys at or above it in the first tiles, and
                                             // those tiles' elements (sums over the cluster)
    uint16_t queue[WARPS][QCAP];             // per-warp vector queues (tile positions)
    unsigned long long full[NSTAGE];         // stage mbarriers
};

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
    uint32_t row_T = 0;      // the row's k-th key once selected (0: none)
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
            if (pass && TOPK_IDX_OK(q + __popc(b & lt), QCAP))
                s->queue[warp][q + __popc(b & lt)] = static_cast<uint16_t>(j * THREADS + static_cast<int>(threadIdx.x));
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
                    if (key >= lim && TOPK_IDX_OK(at, CAP)) {
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

    // Token mode: append every key >= lim of the tile, with packed BF16
    // compares: a non-NaN value x has key(x) >= lim exactly when x >= value(lim)
    // as a BF16 number, for lim in [key(-inf), key(+inf)], except lim = key(+0),
    // where -0 compares equal to +0 and is masked out apart. Below key(-inf)
    // every eligible key qualifies, above key(+inf) none.
    // Each thread forms the 8-bit masks of its vectors. The warp reserves the
    // slots of all its survivors with one
    // shared atomic (a ballot prefix of the counts, or a shuffle scan when a
    // count exceeds 15), then each lane writes its own, reading the values
    // back from the stage. Returns false if the buffer could not take them
    // (the warp's slots are then dead and the warp redoes its part after a
    // compaction), true otherwise.
    __device__ __forceinline__ bool append_masks(const uint4 *stg, int64_t tile_v0, int nv, uint32_t lim) {
        const uint32_t lane = lane_id(), tid = threadIdx.x;
        const uint32_t lo = max(lim, KEY_NEG_INF);
        const bool negz = lo == 0x8000u;  // keys >= key(+0): values >= 0 but -0
        const uint32_t v = lo > KEY_POS_INF ? 0x7FC0u : key_value(lo), cv = v | (v << 16);
        uint32_t mw[2] = {0u, 0u};  // bit 8 (j % 4) + b of word j / 4: vector j's logit 2 (b & 3) + (b >> 2)
        // Every vector's mask, with no branch between them: the loads and the
        // compares of the eight vectors overlap.
        if (!negz) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int pos = j * THREADS + static_cast<int>(tid);
                const uint4 r = pos < nv ? stg[pos] : make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
                mw[j / 4] |= mask8(r, cv) << (8 * (j % 4));
            }
        } else {  // (rare) keys >= key(+0): -0 halves out
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int pos = j * THREADS + static_cast<int>(tid);
                const uint4 r = pos < nv ? stg[pos] : make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
                const uint32_t t = (__vcmpeq2(r.x, 0x80008000u) & 0x00010001u) |
                                   (__vcmpeq2(r.y, 0x80008000u) & 0x00020002u) |
                                   (__vcmpeq2(r.z, 0x80008000u) & 0x00040004u) |
                                   (__vcmpeq2(r.w, 0x80008000u) & 0x00080008u);
                mw[j / 4] |= (mask8(r, cv) & ~((t | (t >> 12)) & 0xFFu)) << (8 * (j % 4));
            }
        }
        const uint32_t cnt = __popc(mw[0]) + __popc(mw[1]);
        uint32_t total, before;
        if (__ballot_sync(0xFFFFFFFFu, cnt > 15u) == 0u) {
            before = warp_excl_small(cnt, total);
        } else {
            const uint32_t incl = warp_incl_scan(cnt);
            before = incl - cnt;
            total = __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (total == 0u) return true;
        uint32_t at;
        if (!reserve(total, before, cnt, at)) return false;
        const uint16_t *h16 = reinterpret_cast<const uint16_t *>(stg);
        const uint32_t i0 = static_cast<uint32_t>(tile_v0) * 8u;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
#pragma unroll 1
            for (uint32_t mm = mw[w]; mm; mm &= mm - 1u) {
                const uint32_t bit = static_cast<uint32_t>(__ffs(mm) - 1);
                const uint32_t j = 4u * w + (bit >> 3), b = bit & 7u;
                const uint32_t h = (j * THREADS + tid) * 8u + 2u * (b & 3u) + (b >> 2);
                if (!TOPK_IDX_OK(h, static_cast<uint32_t>(nv) * 8u) || !TOPK_IDX_OK(at, CAP)) continue;
                const uint32_t key = value_key(h16[h]);
                s->buf_key[at] = static_cast<uint16_t>(key);
                s->buf_idx[at] = i0 + h;
                if (run_ok) atomicAdd(&s->hwin[1][min(key - run_lo, 255u)], 1u);
                ++at;
            }
        }
        (void)lane;
        return true;
    }

    // A carried threshold g for this row, checked on the first tile of every
    // CTA of the cluster before anything is appended: the keys >= g there,
    // scaled to the row's length, must come to between k and 8k (fewer: g is
    // likely above the row's k-th key; more: the buffer would churn). Either
    // way the row then goes on without g, from this same tile. An estimate
    // only: a row that passes and still has fewer than k keys >= g is caught
    // at the end (and streamed again). The same answer on every CTA of the
    // cluster (sums over it, one cluster barrier).
    __device__ __forceinline__ bool guess_holds(const uint4 *stg, int64_t tile_v0, int nv, uint32_t g) {
        const int tid = threadIdx.x;
        mask_tail(stg, tile_v0, nv);  // (this thread's own vector; filter_tile repeats it)
        uint32_t cnt = 0;
        if constexpr (M::BLOCK) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int pos = j * THREADS + tid;
                if (pos < nv) cnt += BlockMode::key(stg[pos], tile_v0 + pos, V) >= g;
            }
        } else {
            uint32_t lo = max(g, KEY_NEG_INF);
            const uint32_t cv = cut_operand(lo);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int pos = j * THREADS + tid;
                cnt += __popc(mask8(pos < nv ? stg[pos] : make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu,
                                                                   0xFFFFFFFFu), cv));
            }
        }
        uint32_t total;
        block_incl_scan(cnt, total);
        const uint32_t elems = static_cast<uint32_t>(
            M::BLOCK ? nv : min(static_cast<int64_t>(nv) * 8, static_cast<int64_t>(L) - 8 * tile_v0));
        uint64_t sum_cnt = total, sum_el = elems;
        if (C > 1) {
            if (tid == 0) {
                red_add_peer(peer_addr(&s->guess_cnt, 0u), total);
                red_add_peer(peer_addr(&s->guess_nv, 0u), elems);
            }
            cluster_arrive();
            cluster_wait();
            sum_cnt = ld_peer(peer_addr(&s->guess_cnt, 0u));
            sum_el = ld_peer(peer_addr(&s->guess_nv, 0u));
        }
        const uint64_t row_el = M::BLOCK ? static_cast<uint64_t>(V) : static_cast<uint64_t>(L);
        const uint64_t est = sum_el ? sum_cnt * row_el / sum_el : 0u;
        return est >= k && est <= 8ull * k;
    }

    // Token mode: the row's last vector, when partial, gets 0xFFFF (a NaN: no
    // cut selects it, no maximum prefers it, its key is 0) in the lanes past
    // the valid length, by the thread that owns its position in this tile (its
    // warp reads it after a warp barrier).
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
                w[h >> 1] |= (h & 1) ? 0xFFFF0000u : 0x0000FFFFu;
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
                        if (!TOPK_IDX_OK(first + r, CAP)) continue;
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
        if (!M::BLOCK && !p->force_direct && nE / 8u >= 2u * k && vector_cut(stg, tile_v0, nv)) return;
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

    // Token rows: first_cut with every vector (8 logits) a group, its
    // representative the largest of its logits (an element of the vector: the
    // packed maximum returns one of its operands and skips NaN halves), all of
    // them held in registers after one pass over the stage. The same window
    // as first_cut's; returns false, with nothing changed, when the k-th
    // largest representative lies below the window (first_cut's general path
    // then takes the row).
    __device__ __forceinline__ bool vector_cut(const uint4 *stg, int64_t tile_v0, int nv) {
        const int tid = threadIdx.x;
        PhaseClock clk;
        clk.start(*p);
        mask_tail(stg, tile_v0, nv);  // this thread's own vector, read back below
        uint32_t rk[VPT];
        uint32_t top = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int pos = j * THREADS + tid;
            rk[j] = pos < nv ? top_key(vec_bmax(stg[pos])) : 0u;
            top = max(top, rk[j]);
        }
        top = __reduce_max_sync(0xFFFFFFFFu, top);
        if (lane_id() == 0) s->red[parity][tid >> 5] = top;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < WARPS; ++w) top = max(top, s->red[parity][w]);
        parity ^= 1u;
        if (top == 0u) return false;
        // Bins of two keys below the top (bin 255: top - 1, top); lower keys
        // are not counted, so a k-th representative below the window shows as
        // too few representatives.
#pragma unroll
        for (int j = 0; j < VPT; ++j)
            if (rk[j] != 0u && top - rk[j] < 510u) atomicAdd(&s->hwin[2][255u - ((top - rk[j]) >> 1)], 1u);
        __syncthreads();
        uint32_t b, wabove, wtotal;
        const bool ok = find_bin256(s->hwin[2], k, b, wabove, wtotal);
        const uint32_t in_bin = ok ? s->hwin[2][b] : 0u;
        __syncthreads();
        s->hwin[2][tid] = 0u;
        __syncthreads();
        if (!ok) return false;
        const uint32_t upper = top - 2u * (255u - b);  // bin b: keys upper - 1, upper
        uint32_t c = upper > 1u ? upper - 1u : 1u;
        if (in_bin > k / 4u) {  // a crowded bin: c exactly the k-th representative
            uint32_t mine = 0;
#pragma unroll
            for (int j = 0; j < VPT; ++j) mine += rk[j] == upper;
            uint32_t ups;
            block_incl_scan(mine, ups);
            if (wabove + ups >= k) c = upper;
        }
        count_event(*p, TOPK_CNT_TILE_SAMPLED);
        first_c = c;
        thr = max(thr, c + 1u);
        publish(c);
        clk.stop(*p, TOPK_CNT_CYC_CUT);
        return true;
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
                if (sel && TOPK_IDX_OK(at, n)) {
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
        // Each thread counts its entries (tid, tid + THREADS, ...) above T and
        // tied at T, packed (ties << 16) | above (n <= CAP < 2^16); one CTA
        // scan gives every thread its first output slot and tie slot, and a
        // second pass writes them: no atomic per entry or per warp.
        uint32_t cnt = 0;
        for (uint32_t i = tid; i < n; i += THREADS) {
            const uint32_t key = s->buf_key[i];
            cnt += key > T ? 1u : (take != 0u && key == T ? 0x10000u : 0u);
        }
        uint32_t total;
        const uint32_t excl = block_incl_scan(cnt, total) - cnt;
        uint32_t ag = excl & 0xFFFFu, at = excl >> 16;
        for (uint32_t i = tid; i < n; i += THREADS) {
            const uint32_t key = s->buf_key[i];
            if (key > T) {
                if (TOPK_IDX_OK(offset + ag, k)) orow[ag] = transform(*p, row, static_cast<int32_t>(s->buf_idx[i]));
                ++ag;
            } else if (take != 0u && key == T) {
                if (at < static_cast<uint32_t>(TIECAP)) s->tie_idx[at] = s->buf_idx[i];
                ++at;
            }
        }
        const uint32_t ngt = total & 0xFFFFu, e = total >> 16;
        if (take == 0u) return ngt;
        __syncthreads();  // every tie index is written
        if (e <= static_cast<uint32_t>(TIECAP)) {
            if (static_cast<uint32_t>(tid) < e) {
                const uint32_t mine = s->tie_idx[tid];
                uint32_t r = 0;
                if (take < e)
                    for (uint32_t u = 0; u < e; ++u) r += s->tie_idx[u] < mine;
                else
                    r = static_cast<uint32_t>(tid);
                if (r < take && TOPK_IDX_OK(offset + ngt + r, k)) orow[ngt + r] = transform(*p, row, static_cast<int32_t>(mine));
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
            if (sel && TOPK_IDX_OK(offset + ngt + at, k)) orow[ngt + at] = transform(*p, row, static_cast<int32_t>(s->buf_idx[i]));
        }
        return ngt + min(take, e);
    }

    // The largest key of buffer entries [0, n) (0 for none), in every thread.
    // (Callers order the buffer's writes before it with a barrier.)
    __device__ __forceinline__ uint32_t buffer_max(uint32_t n) {
        uint32_t m = 0;
        for (uint32_t i = threadIdx.x; i < n; i += THREADS) m = max(m, static_cast<uint32_t>(s->buf_key[i]));
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane_id() == 0) s->red[parity][threadIdx.x >> 5] = m;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < WARPS; ++w) m = max(m, s->red[parity][w]);
        parity ^= 1u;
        return m;
    }

    // The k-th largest key T of buffer entries [0, n) and the count above it,
    // given a lower bound LB >= 1 of T, when every key >= LB lies within 255 of
    // it: one histogram of those keys only (the buffer's stale entries below LB
    // are skipped). Returns false when a key lies further up or fewer than k
    // keys reach LB (the caller then takes window_select). Uses s->hwin[2]
    // (zero on entry and on exit).
    __device__ __forceinline__ bool bound_select(uint32_t n, uint32_t LB, uint32_t *T_out, uint32_t *above_out) {
        const int tid = threadIdx.x;
        bool wide = false;
        for (uint32_t i = tid; i < n; i += THREADS) {
            const uint32_t key = s->buf_key[i];
            if (key >= LB) {
                if (key - LB > 255u) wide = true;
                else atomicAdd(&s->hwin[2][key - LB], 1u);
            }
        }
        const bool any_wide = __syncthreads_or(wide) != 0;
        uint32_t b = 0, above = 0, total;
        const bool ok = !any_wide && find_bin256(s->hwin[2], k, b, above, total);
        __syncthreads();
        s->hwin[2][tid] = 0u;
        __syncthreads();
        *T_out = LB + b;
        *above_out = above;
        return ok;
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
        if (!bound_select(n, max(thr, 2u) - 1u, &T, &above))  // thr - 1: see emit_single
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
        mask_tail(stg, tile_v0, nv);
        clk.stop(*p, TOPK_CNT_CYC_F_PREP);
        clk.start(*p);
        // Token rows: packed masks, the warp's whole part of the tile as one
        // entry (Q = 1); block rows: a queue of candidate vectors.
        uint32_t Q, next;
        if constexpr (!M::BLOCK) {
            Q = 1u;
            next = append_masks(stg, tile_v0, nv, lim) ? 1u : 0u;
        } else {
            Q = build_queue(stg, tile_v0, nv, lim);
            clk.stop(*p, TOPK_CNT_CYC_F_QUEUE);
            clk.start(*p);
            next = append_keys(stg, tile_v0, Q, 0, lim);
        }
        buf_lo = min(buf_lo, lim);
        f_Q = Q;
        f_next = next;
        f_lim = lim;
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
            if constexpr (!M::BLOCK) next = next < f_Q ? (append_masks(stg, tile_v0, nv, lim) ? 1u : 0u) : next;
            else next = append_keys(stg, tile_v0, f_Q, next, lim);
            if (tid == 0) s->v_flag = 0u;
            __syncthreads();
            if (next < f_Q && lane_id() == 0) s->v_flag = 1u;
            __syncthreads();
            if (s->v_flag == 0u) break;  // uniform
        }
    }

    // C == 1: the buffer holds the row's candidates; write its top-k.
    // guessed: the row started from a carried threshold; with fewer than k
    // keys at or above it, nothing is written and false is returned (the row
    // is streamed again without it).
    __device__ __forceinline__ bool emit_single(bool guessed) {
        s->hwin[1][threadIdx.x] = 0u;  // the index radix's scratch (ordered by the barriers below)
        run_ok = false;
        __syncthreads();
        const uint32_t n = min(s->v_count, static_cast<uint32_t>(CAP));
        if (guessed && n < k) return false;
        uint32_t T = 0, take = 0;
        if (n > k) {
            // thr - 1 bounds the buffer's k-th key from below (thr is one above a
            // cut, a compaction's k-th key or a find's F), and so does the last
            // tile's find (v_newthr - 1).
            const uint32_t LB = max(max(thr, s->v_newthr), 2u) - 1u;
            uint32_t above;
            if (!bound_select(n, LB, &T, &above))
                window_select(0, n, buf_lo, max(buffer_max(n), buf_lo), k, &T, &above);
            take = k - above;
            row_T = T;
        }
        const uint32_t written = emit_selected(n, T, take, 0);
        int32_t *orow = p->out + static_cast<int64_t>(row) * k;
        for (uint32_t i = written + threadIdx.x; i < k; i += THREADS) orow[i] = -1;
        return true;
    }

    // Cluster merge: the C buffers (each its CTA's top-k) give the row's k-th
    // key; ties at it go to the lowest indices, lower-ranked CTAs first.
    // guessed: as emit_single (the cluster-wide count decides, the same on
    // every CTA of the cluster).
    __device__ __forceinline__ bool merge_and_emit(bool guessed) {
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
        const bool missed = guessed && !enough;
        if (!missed) {
            // This CTA's part: keys > T, and its quota of the lowest-index ties.
            const uint32_t quota = take > eq_prev ? take - eq_prev : 0u;
            const uint32_t offset = gt_prev + min(eq_prev, take);
            if (!enough) {
                emit_selected(n, LB - 1u, 0u, offset);  // every key >= LB
            } else {
                emit_selected(n, T, quota, offset);
                row_T = T;
            }
            const uint32_t selected_total = enough ? k : total;
            int32_t *orow = p->out + static_cast<int64_t>(row) * k;
            for (uint32_t i = selected_total + rank + static_cast<uint32_t>(tid) * C; i < k; i += THREADS * C)
                orow[i] = -1;
        }
        cluster_wait();
        // Every peer is done with this row's shared words: reset them for the
        // row after next (the next row uses the other parity).
        s->h_merge[0][tid] = 0u;
        s->h_merge[1][tid] = 0u;
        if (tid == 0) {
            s->shared_thr[slot] = 0u;
            s->shared_max[slot] = 0u;
        }
        return !missed;
    }
};

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
        s.guess_cnt = s.guess_nv = 0u;
    }
    for (int i = 0; i < 4; ++i) s.hwin[i][tid] = 0u;
    s.h_merge[0][tid] = s.h_merge[1][tid] = 0u;
    __syncthreads();
    grid_dependency_wait();
    if (p.release) grid_dependents_release();
    Feed feed;
    // One row per cluster at most: a row that misses its carried threshold is
    // streamed again (the ring has nothing of another row in flight).
    const bool one_row = ncl >= p.rows;
    const uint32_t carry_tag = (M::BLOCK ? 0x80000000u : 0u) | (static_cast<uint32_t>(p.k) << 16);
    if (tid == 0) {
        feed_seek(feed, p, M::BLOCK, cid, ncl, C, rank);
        for (int i = 0; i < NSTAGE && feed.row < p.rows; ++i) feed_issue(feed, s, i, p, M::BLOCK, ncl, C, rank);
        // Read once, by rank 0, so that the whole cluster starts from the same
        // word whatever other launches write meanwhile.
        if (rank == 0) s.carry_word = one_row && !p.force_direct ? g_stream_carry[cid % STREAM_CARRY_SLOTS] : 0u;
    }
    if (C > 1) {
        // Every CTA of the cluster has started and zeroed its shared words
        // before any distributed shared memory access.
        cluster_arrive();
        cluster_wait();
    } else {
        __syncthreads();
    }
    uint32_t guess = 0;  // the carried threshold (0: none), the same on every CTA of the cluster
    {
        const uint32_t cw = C > 1 ? ld_peer(peer_addr(&s.carry_word, 0u)) : s.carry_word;
        if ((cw & STREAM_CARRY_TAG_MASK) == carry_tag && !(cw & STREAM_CARRY_DROPPED) &&
            (cw & 0xFFFFu) > STREAM_CARRY_MARGIN)
            guess = (cw & 0xFFFFu) - STREAM_CARRY_MARGIN;
    }
    uint32_t last_T = 0;
    bool dropped = false;  // a row of this cluster dropped its carried threshold

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
        // (V >= C: every CTA of the cluster has a share, so every one checks
        // the threshold on its first tile and meets the others there)
        bool guessed = guess != 0u && V >= static_cast<int64_t>(C);
        for (;;) {  // (twice only when a carried threshold misses)
        cta.row = row;
        cta.L = L;
        cta.V = V;
        cta.thr = guessed ? max(guess, static_cast<uint32_t>(M::KMIN)) : M::KMIN;
        cta.buf_lo = 0xFFFFu;
        cta.best_T = 0;
        cta.row_T = 0;
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
                if (guessed && !cta.guess_holds(stg, tile_v0, nv, guess)) {
                    guessed = false;  // the row goes on without the carried threshold
                    dropped = true;
                    cta.thr = M::KMIN;
                    if (rank == 0) count_event(p, TOPK_CNT_GUESS_MISS);
                }
                cta.thr = max(cta.thr, cta.effective_thr());
                if (!guessed) cta.first_cut(stg, tile_v0, nv);
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
        const bool done = C == 1 ? cta.emit_single(guessed) : cta.merge_and_emit(guessed);
        __syncthreads();
        fin.stop(p, TOPK_CNT_CYC_FINISH);
        if (guessed && rank == 0) count_event(p, done ? TOPK_CNT_GUESS_HIT : TOPK_CNT_GUESS_MISS);
        if (done) break;
        // The carried threshold missed (fewer than k keys at or above it):
        // stream the row again without it, with the other parity's shared
        // words. Every thread is past its last read of the stages.
        guessed = false;
        dropped = true;
        ++it;
        if (tid == 0) {
            fence_proxy_async();
            feed_seek(feed, p, M::BLOCK, row, ncl, C, rank);
            for (int i = 0; i < NSTAGE && feed.row == row; ++i)
                feed_issue(feed, s, static_cast<int>((seq + i) % NSTAGE), p, M::BLOCK, ncl, C, rank);
        }
        cta.snapshot_shared();
        __syncthreads();
        }
        if (cta.row_T != 0u) last_T = cta.row_T;
    }
    if (rank == 0 && tid == 0 && last_T != 0u && !p.force_direct)
        g_stream_carry[cid % STREAM_CARRY_SLOTS] = carry_tag | (dropped ? STREAM_CARRY_DROPPED : 0u) | last_T;
}

constexpr int WIDE_NSTAGE = 2, WIDE_CAP = 4096;

Variant stream_variant(bool block) {
    return block ? Variant{reinterpret_cast<const void *>(&topk_kernel<BlockMode, WIDE_NSTAGE, WIDE_CAP>),
                           static_cast<int>(sizeof(Smem<WIDE_NSTAGE, WIDE_CAP>))}
                 : Variant{reinterpret_cast<const void *>(&topk_kernel<TokenMode, WIDE_NSTAGE, WIDE_CAP>),
                           static_cast<int>(sizeof(Smem<WIDE_NSTAGE, WIDE_CAP>))};
}

cudaError_t status_stream(uint32_t *v, bool clear) { return unit_status(v, clear); }

}  // namespace topk
