// Exact per-row top-k of BF16 logits for GB300 (sm_103a): the one-tile kernel,
// for rows whose valid prefix fits one 32 KiB stage (16384 logits).
//
// The operation: vLLM "decode_topk_cute", module docstring ("What this module
// computes"); the order key and NaN rule: sglang PR #39305 "Exact bf16 consumer
// top-k adapted from DeepSelect", Modifications; lowest-index ties and the
// block-table transform: vLLM kimi_k3 "dsa/indexer", IndexerSelect.
//
// A CTA is persistent over rows; a row arrives by one bulk copy into a 32 KiB
// shared stage. Per row:
//   1. a cut c with at least k keys >= c (so c is at most the k-th key): the
//      cut that held on the CTA's previous row (for its first row, the one its
//      slot ended the last launch with), or the k-th largest of group
//      representatives;
//   2. survivors: every thread forms the 8-bit masks of its vectors' logits
//      >= c with packed BF16 compares (NaN never passes), takes its slots from
//      a warp scan of the counts and one shared atomic per warp, and appends
//      (key << 16 | 0xFFFF - index) words to a list, reading each survivor back
//      from the stage; each survivor is counted in a 256-bin window histogram
//      (bin key - c);
//   3. the k-th key T from the window (one warp), with the counts above it and
//      at it; from here on only the list is read, so the stage takes the next
//      row's copy at once;
//   4. output by one CTA scan of (keys above T, ties at T) counts per thread:
//      every thread writes its selected entries at its scanned slots (no
//      per-key atomics); ties are ranked by index only when not all are taken.
// Fallbacks keep it exact: too few or too many survivors drop the carried cut
// for the representatives' cut, then the exact cut (every key its own
// representative); a crowd of ties beyond the list is written by index-ordered
// rescans of the row.

#include <mutex>

#include "common.cuh"

namespace topk {

namespace one {

// The cut each CTA slot ended its last launch with, per device: (k << 16) |
// cut, bit 31 set for block rows (0: none). A launch's CTA starts from it when
// k and the mode match (decode steps see rows alike from one step to the
// next), so its first row usually skips the representatives' pass. Only a
// starting point: the survivor pass counts exactly the keys at or above any
// cut it tries and falls back on a miss, so results never depend on it.
// Launches running at once (other streams) may overwrite each other's words:
// a 32-bit store is indivisible, and any value is a valid starting point.
constexpr int CARRY_SLOTS = 1024;
static __device__ uint32_t g_carry[CARRY_SLOTS];

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
static constexpr int TAB_CAP = 256;          // page ids of a row staged in shared memory
static constexpr int TPT = (TAB_CAP + NT - 1) / NT;  // page ids per thread
// The build for large k (256 threads, 4096-entry list) also carries the window
// shift of its cuts and measures their distance in value near zero (see
// next_guess): rows that select about half their elements need both. The
// other builds keep the plain distance in keys.
static constexpr bool DENSE_GUESS = NT == 256 && SURV_ == 4096;

struct alignas(128) Smem {
    uint4 stage[NSTAGE][NTILE];
    union {                                  // the representatives are done before survivors start
        uint32_t surv[SURV_CAP + 4];         // (key << 16) | (0xFFFF - index); + a spare slot for
                                             // writes past the end
        uint16_t rep[REP_CAP];               // the row's representatives (0 = none)
    };
    alignas(16) uint32_t hs[4][256];         // [0], [1]: the cut's byte passes (zero between
                                             // uses); [2 + row parity]: the row's window
    alignas(16) uint32_t tie_idx[TIECAP];
    int32_t tab[TAB_CAP];
    uint32_t red[2][NW];
    uint32_t bc[4];
    uint32_t v_cnt[2];                       // survivor counts, by row parity
    uint32_t v_smax;
    uint32_t v_hint;                         // exact_cut: a cut for the next row (see next_guess)
    uint32_t v_carry[NSTAGE];                // a carried cut for the row in each stage (see issue_row)
    uint32_t abort_flag;
    unsigned long long full[NSTAGE];
};

// Histograms are read and written as 16-byte vectors; stages are bulk-copy targets.
static_assert(offsetof(Smem, hs) % 16 == 0 && offsetof(Smem, stage) % 128 == 0, "shared layout");
static_assert(TAB_CAP % NT == 0 || NT % TAB_CAP == 0, "page ids spread evenly over the threads");
static_assert(SURV_CAP < 65536, "scanned counts are packed in 16 bits");

// Inclusive scan over the CTA (one __syncthreads); total = the sum over all.
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
    uint32_t gshift = 0;  // its window's bin width, log2 keys (DENSE_GUESS builds; else 0)
    uint32_t hint = 0;    // exact_cut's cut for the next row (DENSE_GUESS builds; 0: none)
    uint32_t rp = 0;      // parity of the rows this CTA has selected
    bool tab = false;     // the row's page ids are in s.tab
    // The copy ring (thread 0's view): the next row to load into a stage and
    // its valid vectors; the stage of the current row; whether the current
    // row's stage has been handed back to the ring.
    int32_t feed_row = 0, feed_V = 0, step = 1;
    uint32_t *row_carry = nullptr;  // topk_bf16_select_static's per-row cuts (else NULL)
    int32_t cand_row = 0, cand_L = 0;  // the candidate after feed_row and its valid length
                                       // (loaded ahead: nothing waits for it until its turn)
    int st = 0;
    bool fed = false;

    __device__ Row(Smem &s_, const Params &p_) : s(s_), p(p_) {}

    // Vector at position pos: lanes without an element read as 0xFFFF (a NaN:
    // no compare passes it, no maximum prefers it, its key is 0). The row's
    // last vector is masked in place by mask_tail.
    __device__ __forceinline__ uint4 vec(int pos) const {
        if (pos >= V) return make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
        return stg[pos];
    }

    // Token mode: overwrite the lanes of the last vector past the valid length
    // with 0xFFFF, by the thread that owns that position (every later reader of
    // it is that thread or, after a warp barrier, its warp).
    __device__ __forceinline__ void mask_tail() const {
        if (M::BLOCK || (L & 7) == 0 || static_cast<int>(threadIdx.x) != (V - 1) % NT) return;
        const int lanes = L & 7;
        const uint4 r = stg[V - 1];
        uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int h = 0; h < 8; ++h)
            if (h >= lanes) w[h >> 1] |= (h & 1) ? 0xFFFF0000u : 0x0000FFFFu;
        stg[V - 1] = make_uint4(w[0], w[1], w[2], w[3]);
    }

    __device__ __forceinline__ uint32_t bkey(int pos) const {
        return pos < V ? BlockMode::key(stg[pos], pos, V) : 0u;
    }

    __device__ __forceinline__ void clean(int pos, uint32_t (&ck)[4]) const {
        if (pos < V) M::clean(stg[pos], pos, V, L, ck);
        else ck[0] = ck[1] = ck[2] = ck[3] = 0u;
    }

    // Output slot `slot` of the row gets element idx through the transform. A
    // slot past k would break an internal invariant: it is recorded, not written.
    __device__ __forceinline__ void put(uint32_t slot, uint32_t idx) const {
        if (slot >= k) {
            atomicOr(&g_device_status, ERR_BOUNDS);
            return;
        }
        int32_t v = static_cast<int32_t>(idx);
        if (tab) {
            if (!TOPK_IDX_OK(idx >> p.page_shift, TAB_CAP)) return;
            v = s.tab[idx >> p.page_shift] * p.block_rows + (v & ((1 << p.page_shift) - 1));
        }
        else v = transform(p, row, v);
        orow[slot] = v;
    }

    // Representatives of groups of G elements of this thread's vectors
    // j * NT + tid (token: G logits, within a vector for G <= 8, else whole
    // vectors; block: G blocks), fed to f(slot, r, key) in a fixed slot order
    // (r: the thread's r-th representative, slot = r * NT + tid). A token
    // group's representative is its largest logit (0: none, all NaN).
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
                f((2 * j) * NT + tid, 2 * j, top_key(bmax2(r.x, r.y)));
                f((2 * j + 1) * NT + tid, 2 * j + 1, top_key(bmax2(r.z, r.w)));
            }
        } else {
            constexpr int PER = G / 8;  // whole vectors per group
#pragma unroll
            for (int j = 0; j < NV; j += PER) {
                uint32_t acc = vec_bmax(vec(j * NT + tid));
#pragma unroll
                for (int i = 1; i < PER; ++i) acc = bmax2(acc, vec_bmax(vec((j + i) * NT + tid)));
                f((j / PER) * NT + tid, j / PER, top_key(acc));
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
        for (int j = 0; j < NV && j * NT < V; ++j) {  // (vectors past V hold nothing)
            uint32_t ck[4];
            clean(j * NT + tid, ck);
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) {
                const uint32_t key = key_at<M>(ck, h);
                agg_add(s.hs[0], key >> 8, key != 0u);
            }
        }
        __syncthreads();
        if constexpr (DENSE_GUESS) {
            if (tid < 32) {
                // The lowest key of the high byte holding the (k + want)-th
                // largest key: k + want keys at or above it on this row, a cut
                // for the next row counted in ranks; every key (cut 1) when the
                // row has fewer.
                uint32_t b, above, total;
                const bool ok = find_bin256(s.hs[0], k + guess_want(), b, above, total);
                if (tid == 0) s.v_hint = ok ? max(b << 8, 1u) : 1u;
            }
        }
        warp0_find(s, s.hs[0], k);
        __syncthreads();
        if constexpr (DENSE_GUESS) hint = s.v_hint;
        const uint32_t hb = s.bc[0], habove = s.bc[1], nkeys = s.bc[2];
        if (nkeys < k) return false;
        for (int j = 0; j < NV && j * NT < V; ++j) {  // (vectors past V hold nothing)
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
        for (int j = 0; j < NV && j * NT < V; ++j) {  // (vectors past V hold nothing)
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
        for (int j = 0; j < NV && j * NT < V; ++j) {  // (vectors past V hold nothing)
            uint32_t ck[4];
            clean(j * NT + tid, ck);
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) {
                const uint32_t key = key_at<M>(ck, h);
                if (key >= lo && TOPK_IDX_OK(255u - ((top - key) >> 1), 256u))
                    atomicAdd(&s.hs[0][255u - ((top - key) >> 1)], 1u);
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
        for (int j = 0; j < NV && j * NT < V; ++j) {  // (vectors past V hold nothing)
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
    __device__ void take_all(const int32_t (&t0)[TPT]) {
        const int tid = threadIdx.x;
        stage_table(t0);
        uint32_t cnt = 0;
        for (int j = 0; j < NV && j * NT < V; ++j) {  // (vectors past V hold nothing)
            uint32_t ck[4];
            clean(j * NT + tid, ck);
#pragma unroll
            for (int h = 0; h < M::KPV; ++h) cnt += key_at<M>(ck, h) != 0u;
        }
        uint32_t total;
        uint32_t at = block_scan(s, par, cnt, total) - cnt;
        for (int j = 0; j < NV && j * NT < V; ++j) {  // (vectors past V hold nothing)
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
                // (entries past e read as never-smaller; TIECAP is a multiple of 4)
                const uint32_t mine = s.tie_idx[tid];
                uint32_t r = 0;
                for (uint32_t u = 0; u < e; u += 4) {
                    const uint4 t4 = *reinterpret_cast<const uint4 *>(&s.tie_idx[u]);
                    r += (t4.x < mine) + (u + 1 < e && t4.y < mine) + (u + 2 < e && t4.z < mine) +
                         (u + 3 < e && t4.w < mine);
                }
                if (r < take) put(first + r, mine);
            }
            return;
        }
        uint32_t before = 0;
        for (int j = 0; j < NV && j * NT < V && before < take; ++j) {
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

    // The q-th largest of the list's keys in [lo, hi] (others are not
    // counted; q at most their number), by a radix select over the list: one
    // pass when hi - lo < 256, else two.
    __device__ uint32_t survivor_select(uint32_t n, uint32_t lo, uint32_t hi, uint32_t q, uint32_t &above) {
        const uint32_t tid = threadIdx.x;
        const uint32_t range = hi - lo;
        const int shift = range < 256u ? 0 : (32 - __clz(static_cast<int>(range))) - 8;
        const uint32_t mask = (1u << shift) - 1u;
        for (uint32_t i = tid; i < n; i += NT) {
            const uint32_t o = (s.surv[i] >> 16) - lo;  // (keys below lo wrap past range)
            if (o <= range) atomicAdd(&s.hs[0][min(o >> shift, 255u)], 1u);
        }
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
            const uint32_t o = (s.surv[i] >> 16) - lo;
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

    // Token rows: survivors of cut c (cv = cut_operand(c)): every key >= c
    // goes to the list as (key << 16) | (0xFFFF - index), and to the window
    // histogram hw (bin key - c, the top bin holding every key >= c + 255).
    // Each thread forms the 8-bit masks of all its vectors with packed BF16
    // compares (independent, so they overlap), packed into one 64-bit word;
    // slots come from a ballot prefix of the counts and one shared atomic per
    // warp; then one loop over the thread's survivors reads each back from the
    // stage as a 16-bit value (no per-vector loops, no register indexing).
    __device__ __forceinline__ void survivors_tok(uint32_t c, uint32_t cv, uint32_t *hw, uint32_t sh) {
        constexpr int MW = (NV + 3) / 4;  // mask words: bit 8 (j % 4) + b of word j / 4 is
                                          // vector j's logit 2 (b & 3) + (b >> 2)
        const uint32_t lane = lane_id(), tid = threadIdx.x;
        uint32_t mw[MW] = {};
#pragma unroll
        for (int j = 0; j < NV; ++j) mw[j / 4] |= mask8(vec(j * NT + static_cast<int>(tid)), cv) << (8 * (j % 4));
        uint32_t cnt = 0;  // <= 8 NV
#pragma unroll
        for (int w = 0; w < MW; ++w) cnt += __popc(mw[w]);
        const uint32_t lt = (1u << lane) - 1u;
        (void)lt;
        const uint32_t incl = warp_incl_scan(cnt);
        const uint32_t before = incl - cnt, tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        uint32_t base = 0;
        if (lane == 0 && tot) base = atomicAdd(&s.v_cnt[rp], tot);
        uint32_t at = __shfl_sync(0xFFFFFFFFu, base, 0) + before;
        const uint16_t *h16 = reinterpret_cast<const uint16_t *>(stg);
#pragma unroll
        for (int w = 0; w < MW; ++w) {
#pragma unroll 1
            for (uint32_t mm = mw[w]; mm; mm &= mm - 1u) {
                const uint32_t bit = static_cast<uint32_t>(__ffs(mm) - 1);
                const uint32_t j = 4u * w + (bit >> 3), b = bit & 7u;
                const uint32_t idx = (j * NT + tid) * 8u + 2u * (b & 3u) + (b >> 2);
                if (!TOPK_IDX_OK(idx, static_cast<uint32_t>(V) * 8u)) continue;
                const uint32_t key = value_key(h16[idx]);
                // Past the list's end (the count then exceeds it and the pass is
                // redone or replaced) writes go to the spare slot.
                s.surv[min(at, static_cast<uint32_t>(SURV_CAP))] = (key << 16) | (0xFFFFu - idx);
                atomicAdd(&hw[min((key - c) >> sh, 255u)], 1u);
                ++at;
            }
        }
    }

    // Block rows: survivors of cut c, as survivors_tok with one key per vector
    // (bit j: vector j's key >= c; the key is formed again for the write).
    __device__ __forceinline__ void survivors_blk(uint32_t c, uint32_t *hw, uint32_t sh) {
        const uint32_t tid = threadIdx.x;
        uint32_t m = 0, cnt = 0;
#pragma unroll
        for (int j = 0; j < NV; ++j)
            if (bkey(j * NT + static_cast<int>(tid)) >= c) m |= 1u << j;
        cnt = __popc(m);
        const uint32_t incl = warp_incl_scan(cnt);
        const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        uint32_t base = 0;
        if (lane_id() == 0 && tot) base = atomicAdd(&s.v_cnt[rp], tot);
        uint32_t at = __shfl_sync(0xFFFFFFFFu, base, 0) + incl - cnt;
#pragma unroll 1
        for (; m; m &= m - 1u) {
            const uint32_t idx = static_cast<uint32_t>(__ffs(m) - 1) * NT + tid;
            const uint32_t key = bkey(static_cast<int>(idx));
            s.surv[min(at, static_cast<uint32_t>(SURV_CAP))] = (key << 16) | (0xFFFFu - idx);
            atomicAdd(&hw[min((key - c) >> sh, 255u)], 1u);
            ++at;
        }
    }

    // Output of the list (n entries) given the k-th key T, the count above it
    // and the ties to take: one CTA scan of each thread's (above T, equal to T)
    // counts gives every selected entry its slot, keys above T first. Ties go
    // straight to their slots when all of them are taken; otherwise they are
    // ranked by index (write_ties).
    __device__ __forceinline__ void emit(uint32_t n, uint32_t T, uint32_t above, uint32_t take) {
        const uint32_t tid = threadIdx.x;
        const uint32_t lo_e = T << 16, hi_e = (T + 1u) << 16;  // entries of key T: [lo_e, hi_e)
        uint32_t cnt = 0;  // (ties << 16) | above, this thread's entries tid + u NT
        for (uint32_t i0 = tid; i0 < n; i0 += 4u * NT) {
            uint32_t x[4];  // four entries loaded together (0: none)
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = i0 + u * NT < n ? s.surv[i0 + u * NT] : 0u;
#pragma unroll
            for (int u = 0; u < 4; ++u) cnt += x[u] >= hi_e ? 1u : x[u] >= lo_e ? 0x10000u : 0u;
        }
        uint32_t total;
        const uint32_t pre = block_scan(s, par, cnt, total) - cnt;
        const uint32_t e = total >> 16;  // the ties at T (and total & 0xFFFF == above)
        const bool all = take == e;
        uint32_t a_at = pre & 0xFFFFu, t_at = pre >> 16;
        for (uint32_t i0 = tid; cnt != 0u && i0 < n; i0 += 4u * NT) {
            uint32_t x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = i0 + u * NT < n ? s.surv[i0 + u * NT] : 0u;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t idx = 0xFFFFu - (x[u] & 0xFFFFu);
                if (x[u] >= hi_e) {
                    put(a_at++, idx);
                } else if (x[u] >= lo_e) {
                    if (all) put(above + t_at, idx);
                    else if (t_at < static_cast<uint32_t>(TIECAP)) s.tie_idx[t_at] = idx;
                    ++t_at;
                }
            }
        }
        if (!all) {
            __syncthreads();
            write_ties(T, take, above, e);
        }
    }

    // The exact cut c with more keys at or above it than the list holds (a
    // crowd of ties at c): keys > c in index order, then the lowest-index ties.
    __device__ void emit_rescan(uint32_t c) {
        const int tid = threadIdx.x;
        uint32_t before = 0;
        for (int j = 0; j < NV && j * NT < V; ++j) {  // (vectors past V hold nothing)
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
    //
    // DENSE_GUESS builds: around zero BF16 keys step through tiny magnitudes,
    // where a distance in keys says nothing about ranks, so within 1/8 of zero
    // the distance is taken in value; after the exact cut (T = c: no spacing
    // measured) the cut is exact_cut's hint. The next row's window histogram
    // is then binned 2^gshift keys wide, so that T - cut spans at most 127
    // bins (up to 256 keys per bin: the list's radix select places the k-th
    // key inside its bin).
    __device__ __forceinline__ uint32_t guess_want() const {
        return min(max(k / 8u, 128u), (static_cast<uint32_t>(SURV_CAP) - k) / 2u);
    }

    __device__ __forceinline__ void next_guess(uint32_t c, uint32_t T, uint32_t n) {
        const uint32_t want = guess_want();
        uint32_t d = T > c ? max(static_cast<uint32_t>(__fdividef(static_cast<float>(want * (T - c)),
                                                                  static_cast<float>(n - k + 1u))), 1u)
                           : 16u;
        if constexpr (DENSE_GUESS) {
            if (T > c && T - 0x41FFu < 0x7C01u) {  // T's value in [-1/8, 1/8)
                const float vT = __uint_as_float(key_value(T) << 16), vc = __uint_as_float(key_value(c) << 16);
                const float vg = vT - (vT - vc) * __fdividef(static_cast<float>(want), static_cast<float>(n - k + 1u));
                const uint32_t kg = value_key(__float_as_uint(vg) >> 16);  // (the key below covers truncation)
                if (isfinite(vg) && kg > 1u && kg <= T) d = T - (kg - 1u);
            } else if (T <= c && hint != 0u && hint < T) {
                d = T - hint;
            }
            d = min(d, 127u << 8);  // (gshift <= 8)
            gshift = 0u;
            while ((d >> gshift) > 127u) ++gshift;
        }
        guess = T > d ? T - d : 1u;
    }

    // Hand the current row's stage back to the copy ring: thread 0 issues the
    // next row's copy into it. Every thread must be done reading the stage
    // (a barrier since its last read orders those reads before the fence).
    __device__ __forceinline__ void feed() {
        fed = true;
        if (threadIdx.x == 0 && feed_row < p.rows) {
            fence_proxy_async();
            issue_row(s, st, p, feed_row, feed_V, row_carry != nullptr ? row_carry[feed_row] : 0u);
            advance_feed();
        }
    }

    // Thread 0: feed_row = the next row that reads logits (p.rows if none),
    // from the prefetched candidate; then the next candidate's length is
    // loaded ahead.
    __device__ __forceinline__ void advance_feed() {
        for (;;) {
            if (cand_row >= p.rows) {
                feed_row = p.rows;
                return;
            }
            const int32_t L = min(max(cand_L, 0), p.width);
            const int32_t n = M::BLOCK ? (L + 7) >> 3 : L;
            const int32_t r = cand_row;
            cand_row += step;
            if (cand_row < p.rows) cand_L = __ldg(p.valid_len + cand_row);
            if (n > p.k) {
                feed_row = r;
                feed_V = (L + 7) >> 3;
                return;
            }
        }
    }

    // Store the page ids loaded at the start of select() (the caller
    // synchronises before the first put).
    __device__ __forceinline__ void stage_table(const int32_t (&t0)[TPT]) const {
#pragma unroll
        for (int u = 0; u < TPT; ++u)
            if (tab && threadIdx.x + u * NT < static_cast<uint32_t>(TAB_CAP)) s.tab[threadIdx.x + u * NT] = t0[u];
    }

    __device__ void select() {
        const uint32_t tid = threadIdx.x;
        const uint32_t nE = M::BLOCK ? static_cast<uint32_t>(V) : static_cast<uint32_t>(L);
        // The row's page ids, loaded now and staged in shared memory before the
        // first write (their latency hides behind the survivor pass).
        int32_t t0[TPT] = {};  // page ids of this thread's entries tid + u NT
        tab = false;
        if (p.table) {
            const uint32_t npages = (nE + (1u << p.page_shift) - 1u) >> p.page_shift;
            if (npages <= static_cast<uint32_t>(TAB_CAP)) {
                tab = true;
                const int32_t *trow = table_row(p, row);
#pragma unroll
                for (int u = 0; u < TPT; ++u)
                    if (tid + u * NT < npages) t0[u] = __ldg(trow + tid + u * NT);
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
            // (nE / (2 g) >= 2 k written as nE >= 4 g k, all below 2^32)
            if constexpr (M::BLOCK) {
                while (g < min(8u, static_cast<uint32_t>(NV)) && nE >= 4u * g * k) g *= 2u;
            } else {
                g = 4;
                while (g < min(64u, 8u * NV) && nE >= 4u * g * k) g *= 2u;
                if (nE < 2u * g * k) g = 1;  // too few groups of 4: exact path
            }
        }
        // First try the previous row's cut: any c with at least k keys >= c
        // bounds the k-th largest key from below, and the survivor pass counts
        // exactly those keys; a cut with too few of them or more than the list
        // holds is dropped for the representatives' cut.
        bool guessed = guess != 0u && !p.force_direct;
        hint = 0u;
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
            // cs: the cut as the survivor pass applies it (c, or a lower key
            // the packed compares can apply exactly); c stays the cut found.
            uint32_t cs = c;
            const uint32_t cv = cut_operand(cs);
            const uint32_t sh = DENSE_GUESS && guessed ? gshift : 0u;  // the window's bins: 2^sh keys
            if constexpr (M::BLOCK) survivors_blk(cs, hw, sh);
            else survivors_tok(cs, cv, hw, sh);
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
                emit_rescan(c);  // the exact cut (the k-th key), with a crowd of ties at it
                guess = c > 16u ? c - 16u : 1u;
                gshift = 0u;
                clk.stop(p, TOPK_CNT_CYC_FINISH);
                return;
            }
            count_event(p, guessed ? TOPK_CNT_GUESS_HIT : g == 1u ? TOPK_CNT_TILE_EXACT : TOPK_CNT_TILE_SAMPLED);
            if (tid < 32u) {  // warp 0: the k-th key's bin, the count above it and in it
                uint32_t b0, a0, t0w;
                find_bin256(hw, k, b0, a0, t0w);
                if (tid == 0) {
                    s.bc[0] = b0;
                    s.bc[1] = a0;
                    s.bc[3] = hw[b0];
                }
            }
            __syncthreads();
            uint32_t b = s.bc[0], above = s.bc[1];
            uint32_t T = cs + (b << sh), at_T = s.bc[3];
            if (sh != 0u && b < 255u) {
                // Wide bins: the k-th key lies in [T, T + 2^sh), which the
                // list's radix select places (its first barrier follows every
                // thread's read of s.bc). The ties at it are not counted: the
                // stage stays until the row is written.
                uint32_t a2;
                T = survivor_select(n, T, T + (1u << sh) - 1u, k - above, a2);
                above += a2;
                at_T = static_cast<uint32_t>(TIECAP) + 1u;
            }
            if (b < 255u && at_T <= static_cast<uint32_t>(TIECAP)) {
                // From here on only the list and the tie buffer are read: the
                // stage takes the next row's copy now, which overlaps the rest.
                feed();
            }
            if (b == 255u) {
                // The k-th key is at least c + 255: find it by radix select over
                // the list.
                uint32_t smax = 0;
                for (uint32_t i = tid; i < n; i += NT) smax = max(smax, s.surv[i] >> 16);
                smax = __reduce_max_sync(0xFFFFFFFFu, smax);
                if (lane_id() == 0) atomicMax(&s.v_smax, smax);
                __syncthreads();
                T = survivor_select(n, cs, s.v_smax, k, above);
                if (tid == 0) s.v_smax = 0u;
            }
            clk.stop(p, TOPK_CNT_CYC_EXACT);
            clk.start(p);
            next_guess(cs, T, n);
            emit(n, T, above, k - above);
            clk.stop(p, TOPK_CNT_CYC_FINISH);
            return;
        }
    }
};

// Thread 0: the copy of a row into stage st, with the carried word for that
// row (0: none) in s.v_carry[st]. The copy's arrival on the stage's barrier
// releases the word, so every thread that waits for the stage reads the same
// one, whatever other launches write to the carry tables meanwhile.
static __device__ __forceinline__ void issue_row(Smem &s, int st, const Params &p, int32_t row, int32_t V,
                                                 uint32_t carried) {
    s.v_carry[st] = carried;
    const uint32_t bytes = static_cast<uint32_t>(V) * 16u;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.logits + static_cast<int64_t>(row) * p.row_stride);
    mbar_expect_tx(&s.full[st], bytes);
    bulk_load(&s.stage[st][0], src, bytes, &s.full[st]);
}

};  // struct Tile

// Carried words: bit 31 block rows, bits 27-30 the cut's window shift
// (DENSE_GUESS builds), bits 16-26 k - 1, bits 0-15 the cut.
static constexpr uint32_t CARRY_TAG_MASK = 0x87FF0000u;

// The kernel's body. row_carry: NULL, or a table of per-row starting cuts
// (carried words) read as each row's copy is issued and rewritten after the
// row (topk_bf16_select_static's variant).
template <class M, int NT, int SURV>
__device__ __forceinline__ void one_tile_body(const Params &p, uint32_t *row_carry) {
    using O = Tile<NT, SURV>;
    constexpr int NSTAGE = O::NSTAGE;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    typename O::Smem &s = *reinterpret_cast<typename O::Smem *>(smem_raw);
    const int tid = threadIdx.x;
    const int32_t step = static_cast<int32_t>(gridDim.x);

    if (tid == 0) {  // (shared-memory set-up before the wait: it touches no global memory)
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

    typename O::template Row<M> r(s, p);
    r.k = static_cast<uint32_t>(p.k);
    const uint32_t carry_tag = (M::BLOCK ? 0x80000000u : 0u) | ((static_cast<uint32_t>(p.k) - 1u) << 16);
    r.step = step;
    r.feed_row = p.rows;
    r.row_carry = row_carry;
    if (tid == 0) {
        r.cand_row = static_cast<int32_t>(blockIdx.x);
        if (r.cand_row < p.rows) r.cand_L = __ldg(p.valid_len + r.cand_row);
        r.advance_feed();
        // The first row carries the cut this CTA slot ended the last launch
        // with (or, static variant, the row's own when it has one for this k).
        uint32_t first = g_carry[blockIdx.x % CARRY_SLOTS];
        for (int i = 0; i < NSTAGE && r.feed_row < p.rows; ++i) {
            uint32_t w = row_carry != nullptr ? row_carry[r.feed_row] : 0u;
            if ((w & CARRY_TAG_MASK) != carry_tag) w = i == 0 ? first : 0u;
            O::issue_row(s, i, p, r.feed_row, r.feed_V, w);
            r.advance_feed();
        }
    }
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
        r.st = st;
        r.fed = false;
        r.orow = p.out + static_cast<int64_t>(row) * p.k;
        PhaseClock clk;
        clk.start(p);
        mbar_wait_sleep(&s.full[st], (seq / NSTAGE) & 1u, &s.abort_flag);
        clk.stop(p, TOPK_CNT_CYC_WAIT);
        {  // the row's carried cut, when it has one for this k and mode (see issue_row)
            const uint32_t cw = s.v_carry[st];
            if ((cw & CARRY_TAG_MASK) == carry_tag && !p.force_direct) {
                r.guess = cw & 0xFFFFu;
                if constexpr (O::DENSE_GUESS) r.gshift = min((cw >> 27) & 15u, 8u);
            }
        }
        count_event(p, TOPK_CNT_ROUNDS);
        ++seq;
        clk.start(p);
        r.select();
        __syncthreads();  // every thread is done with this stage and the row's shared state
        clk.stop(p, TOPK_CNT_CYC_SELECT);
        if (!r.fed) r.feed();
        if (row_carry != nullptr && tid == 0 && r.guess != 0u) row_carry[row] = carry_tag | (r.gshift << 27) | r.guess;
    }
    if (tid == 0 && r.guess != 0u) g_carry[blockIdx.x % CARRY_SLOTS] = carry_tag | (r.gshift << 27) | r.guess;
}

template <class M, int NT, int SURV>
__global__ void __launch_bounds__(NT, NT == 256 ? (SURV <= 2048 ? 4 : 3) : 1) topk_one_tile_kernel(const Params p) {
    one_tile_body<M, NT, SURV>(p, nullptr);
}

// topk_bf16_select_static's kernel: the same, with per-row starting cuts in
// the static table below (its device address is passed in, see
// static_row_carry).
template <class M, int NT, int SURV>
__global__ void __launch_bounds__(NT, NT == 256 ? (SURV <= 2048 ? 4 : 3) : 1)
    topk_one_tile_static_kernel(const Params p, uint32_t *row_carry) {
    one_tile_body<M, NT, SURV>(p, row_carry);
}

// The per-row starting cuts of topk_bf16_select_static: TOPK_STATIC_MAX_ROWS
// words (256 KiB) in every device that loads the library, for the life of the
// process. Hints only (a stale, foreign or raced entry costs speed, never
// correctness), so nothing in it has to start at zero.
static __device__ __align__(256) uint32_t g_row_carry[TOPK_STATIC_MAX_ROWS];

}  // namespace one

template <class M, int NT, int SURV>
static Variant one_build() {
    return Variant{reinterpret_cast<const void *>(&one::topk_one_tile_kernel<M, NT, SURV>),
                   static_cast<int>(sizeof(typename one::Tile<NT, SURV>::Smem))};
}

// build 0: 256 threads, k <= 1024; 1: 256 threads, larger k; 2: 512 threads
// (rows that do not fill the SMs).
Variant one_variant(bool block, int build) {
    switch (build) {
        case 0: return block ? one_build<BlockMode, 256, 2048>() : one_build<TokenMode, 256, 2048>();
        case 1: return block ? one_build<BlockMode, 256, 4096>() : one_build<TokenMode, 256, 4096>();
        default: return block ? one_build<BlockMode, 512, 4096>() : one_build<TokenMode, 512, 4096>();
    }
}

cudaError_t status_one(uint32_t *v, bool clear) { return unit_status(v, clear); }

template <class M, int NT, int SURV>
static Variant one_static_build() {
    return Variant{reinterpret_cast<const void *>(&one::topk_one_tile_static_kernel<M, NT, SURV>),
                   static_cast<int>(sizeof(typename one::Tile<NT, SURV>::Smem))};
}

Variant one_static_variant(bool block, int build) {
    switch (build) {
        case 0: return block ? one_static_build<BlockMode, 256, 2048>() : one_static_build<TokenMode, 256, 2048>();
        case 1: return block ? one_static_build<BlockMode, 256, 4096>() : one_static_build<TokenMode, 256, 4096>();
        default: return block ? one_static_build<BlockMode, 512, 4096>() : one_static_build<TokenMode, 512, 4096>();
    }
}

// Set-up of topk_bf16_select_static on device `dev` (which must be current),
// once per device: the device address of the static table (host code sees
// only a stand-in for it, never to be passed to a kernel) and the kernels'
// shared-memory attribute. Returns the first call's result on every call.
cudaError_t static_row_carry(int dev, uint32_t **table) {
    static std::once_flag once[64];
    static uint32_t *addr[64];
    static cudaError_t err[64];
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev]() {
        void *a = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&a, one::g_row_carry);
        for (int b = 0; b < 2 && e == cudaSuccess; ++b)
            for (int w = 0; w < ONE_BUILDS && e == cudaSuccess; ++w) {
                const Variant v = one_static_variant(b != 0, w);
                e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem);
            }
        addr[dev] = static_cast<uint32_t *>(a);
        err[dev] = e;
    });
    *table = addr[dev];
    return err[dev];
}

}  // namespace topk
