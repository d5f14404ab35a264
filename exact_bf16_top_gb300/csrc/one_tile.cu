// Exact per-row top-k of BF16 logits for GB300 (sm_103a): the one-tile kernel,
// for rows whose valid prefix fits one 32 KiB stage (16384 logits).
//
// The operation: vLLM "decode_topk_cute", module docstring ("What this module
// computes"); the order key and NaN rule: sglang PR #39305 "Exact bf16 consumer
// top-k adapted from DeepSelect", Modifications; lowest-index ties and the
// block-table transform: vLLM kimi_k3 "dsa/indexer", IndexerSelect.

#include "common.cuh"

namespace topk {

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

}  // namespace topk
