// Exact per-row top-k of BF16 logits for GB300 (sm_103a) in ascending index
// order, bounded by the scorer's per-8 maxima (vLLM kimi_k3 "dsa/indexer",
// IndexerSelect), its B' words mode (IndexerLocalTopk), and the per-8 maxima
// kernel.
//
// The operation: vLLM "decode_topk_cute", module docstring ("What this module
// computes"); the order key and NaN rule: sglang PR #39305 "Exact bf16 consumer
// top-k adapted from DeepSelect", Modifications; lowest-index ties and the
// block-table transform: vLLM kimi_k3 "dsa/indexer", IndexerSelect.

#include "common.cuh"

namespace topk {

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

constexpr int NW = NT / 32;
constexpr int REP_CAP = 16384;   // representatives: every top (rows of up to 16384 groups), else
                                 // every piece's maximum (up to 16384 pieces: 1M logits)
constexpr int VEC_CAP = 8192;    // candidate vectors listed
constexpr int KEY_CAP = 8192;    // candidate keys listed
constexpr int STAGE_VECS = (VEC_CAP * 4 + KEY_CAP * 6) / 16;  // rows the exact select keeps in shared memory
constexpr int MAX_BATCHES = 4;   // 256-piece batches of a warp's range of tops (16384 pieces / 16 warps)

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
    if (!TOPK_IDX_OK(slot, p.k)) return;
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
                    if (w.each && TOPK_IDX_OK(8 * pc + e, REP_CAP)) s.rep[8 * pc + e] = static_cast<uint16_t>(top);
                    acc = max(acc, top);
                }
                if (!w.each && TOPK_IDX_OK(pc, REP_CAP)) s.rep[pc] = static_cast<uint16_t>(acc);
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
            for (; m; m &= m - 1u)
                if (TOPK_IDX_OK(pos, VEC_CAP)) s.cvec[pos++] = static_cast<uint32_t>(8 * p0 + __ffsll(m) - 1);
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
                if (!TOPK_IDX_OK(at, KEY_CAP)) continue;
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

Variant ordered_variant() {
    return Variant{reinterpret_cast<const void *>(&ordered::topk_ordered_kernel),
                   static_cast<int>(sizeof(ordered::Smem))};
}

cudaError_t launch_tops(const uint16_t *logits, int64_t row_stride, int32_t rows, int32_t width,
                        const int32_t *valid_len, uint16_t *tops, int64_t tops_stride, int32_t pieces,
                        unsigned blocks, cudaStream_t stream) {
    ordered::topk_tops_kernel<<<blocks, 256, 0, stream>>>(logits, row_stride, rows, width, valid_len, tops,
                                                          tops_stride, pieces);
    return cudaGetLastError();
}

cudaError_t status_ordered(uint32_t *v, bool clear) { return unit_status(v, clear); }

}  // namespace topk
