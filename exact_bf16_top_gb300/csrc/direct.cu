// Exact per-row top-k of BF16 logits for GB300 (sm_103a): the resident-keys
// cluster kernel, for block-mode rows wider than one 32 KiB stage.
//
// The operation: vLLM "decode_topk_cute", module docstring ("What this module
// computes"); the order key and NaN rule: sglang PR #39305 "Exact bf16 consumer
// top-k adapted from DeepSelect", Modifications; lowest-index ties and the
// block-table transform: vLLM kimi_k3 "dsa/indexer", IndexerSelect.

#include "common.cuh"

namespace topk {

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
// representatives cannot bound the k-th key. Before all that, a cluster tries
// the k-th key its slot selected last, less a margin, as c (see g_carry); the
// representatives' histogram is then built only if that cut misses. Used where
// a buffer would churn: block rows, whose k is large next to a CTA's share.

namespace direct {

constexpr int NSTAGE = 2;
// Carried cuts: each cluster slot keeps the k-th key of the last row it
// selected (tagged with the mode and k); its next row, in this launch or the
// next, first tries that key lowered by CARRY_MARGIN as its cut, which the
// row's own window sums then accept or reject (a starting point only).
constexpr int CARRY_SLOTS = 256;
constexpr uint32_t CARRY_MARGIN = 12;
static __device__ uint32_t g_carry[CARRY_SLOTS];
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
    uint32_t carry_word;                     // rank 0: the carried cut this launch starts from
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
    uint32_t kth = 0;    // the row's k-th key once selected (0: none)
    uint32_t guess = 0;  // a carried cut to try first (0: none)

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
                if (!TOPK_IDX_OK(local, RES)) continue;
                s.key[local] = static_cast<uint16_t>(key);
                best = max(best, key);
            } else {
                uint32_t ck[4];
                TokenMode::clean(stg[pos], v, V, L, ck);  // packed pairs of keys, in element order
                if (!TOPK_IDX_OK(local, RES / 8)) continue;
                reinterpret_cast<uint4 *>(s.key)[local] = make_uint4(ck[0], ck[1], ck[2], ck[3]);
                best = max(best, umax_halves(umax2(umax2(ck[0], ck[1]), umax2(ck[2], ck[3]))));
            }
        }
        if (!p.force_direct) {  // (uniform: the exact passes start from an empty h[0])
            if (TOPK_IDX_OK(tile * NT + static_cast<int>(threadIdx.x), MAX_TILES * NT))
                s.rep[tile * NT + static_cast<int>(threadIdx.x)] = static_cast<uint16_t>(best);
            if (guess == 0u) agg_add(s.h[0], best >> 8, best != 0u);  // (else only on a miss)
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
        if (!TOPK_IDX_OK(orow - (p.out + static_cast<int64_t>(row) * p.k) + slot, p.k)) return;
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
            kth = T;
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
        const int r = select_from(c, clk);  // at least k keys are >= c
        if (r != 0) {  // the k-th key is >= c + 255: not resolved by the window
            if (rank == 0) count_event(p, TOPK_CNT_TILE_OVERFLOW);
            return false;
        }
        if (rank == 0) count_event(p, TOPK_CNT_TILE_SAMPLED);
        return true;
    }

    // The selection from a cut c: this CTA's keys >= c listed and binned by
    // key - c, the window summed over the cluster, the k-th key T = c + bin,
    // then the emission. Returns 1 (nothing written) when fewer than k keys of
    // the row reach c, 2 when the k-th key lies past the window (>= c + 255),
    // 0 when done. Every CTA of the cluster returns the same.
    __device__ int select_from(uint32_t c, PhaseClock &clk) {
        const int tid = threadIdx.x;
        const uint32_t k = static_cast<uint32_t>(p.k);
        const uint32_t lane = lane_id();
        list_survivors(c);
        gather(2, 0);
        clk.stop(p, TOPK_CNT_CYC_SURVIVORS);
        clk.start(p);
        uint32_t t, above, tot3;
        if (!find_bin256(s.all, k, t, above, tot3)) return 1;
        if (t == 255u) return 2;
        const uint32_t T = c + t;       // the row's k-th largest key
        kth = T;
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
            return 0;
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
        return 0;
    }

    // The carried cut first: on a miss, every peer is done reading this CTA's
    // window sums before they are cleared, and the row goes on as without it.
    __device__ bool guess_select(uint32_t ntiles, PhaseClock &clk) {
        const int tid = threadIdx.x;
        if (tid == 0) s.n_list = s.cursor[0] = s.cursor[1] = 0u;
        __syncthreads();
        if (select_from(guess, clk) == 0) {
            if (rank == 0) count_event(p, TOPK_CNT_GUESS_HIT);
            return true;
        }
        if (rank == 0) count_event(p, TOPK_CNT_GUESS_MISS);
        if (C > 1) {
            cluster_arrive();
            cluster_wait();
        } else {
            __syncthreads();
        }
        s.h[2][tid] = 0u;
        // The representatives' high bytes, which the stream left out.
        for (uint32_t j = 0; j < ntiles; ++j) {
            const uint32_t r = s.rep[j * NT + static_cast<uint32_t>(tid)];
            agg_add(s.h[0], r >> 8, r != 0u);
        }
        __syncthreads();
        return false;
    }

    __device__ void select_and_emit(uint32_t ntiles) {
        const int tid = threadIdx.x;
        PhaseClock clk;
        clk.start(p);
        bool done = false;
        kth = 0u;
        if (!p.force_direct) {
            if (guess != 0u) done = guess_select(ntiles, clk);
            if (!done) done = cut_select(ntiles, clk);
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
    const uint32_t carry_tag = (M::BLOCK ? 0x80000000u : 0u) | (static_cast<uint32_t>(p.k) << 16);
    if (tid == 0) {
        feed_seek(feed, p, M::BLOCK, cid, ncl, C, rank);
        for (int i = 0; i < NSTAGE && feed.row < p.rows; ++i) feed_issue(feed, s, i, p, M::BLOCK, ncl, C, rank);
        // Read once, by rank 0, so that the whole cluster starts from the same
        // word whatever other launches write meanwhile.
        if (rank == 0) s.carry_word = g_carry[cid % CARRY_SLOTS];
    }
    if (C > 1) {  // every CTA started and zeroed before any distributed access
        cluster_arrive();
        cluster_wait();
    } else {
        __syncthreads();
    }
    Share<M> sh(s, p);
    sh.C = C;
    sh.rank = rank;
    {
        const uint32_t cw = C > 1 ? ld_peer(peer_addr(&s.carry_word, 0u)) : s.carry_word;
        const uint32_t cut = cw & 0xFFFFu;
        if ((cw & 0xFFFF0000u) == carry_tag && cut > CARRY_MARGIN) sh.guess = cut - CARRY_MARGIN;
    }
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
        if (sh.kth > CARRY_MARGIN) sh.guess = sh.kth - CARRY_MARGIN;  // (uniform: from cluster sums)
        __syncthreads();
    }
    if (rank == 0 && tid == 0 && sh.kth != 0u) g_carry[cid % CARRY_SLOTS] = carry_tag | sh.kth;
    whole.stop(p, TOPK_CNT_CYC_KERNEL);
}

}  // namespace direct

Variant direct_variant(bool block) {
    return block ? Variant{reinterpret_cast<const void *>(&direct::topk_direct_kernel<BlockMode>),
                           static_cast<int>(sizeof(direct::Smem))}
                 : Variant{reinterpret_cast<const void *>(&direct::topk_direct_kernel<TokenMode>),
                           static_cast<int>(sizeof(direct::Smem))};
}

cudaError_t status_direct(uint32_t *v, bool clear) { return unit_status(v, clear); }

}  // namespace topk
