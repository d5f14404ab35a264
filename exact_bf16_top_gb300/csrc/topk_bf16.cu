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
// A stage (a "tile": 256 threads x 8 vectors) is handled in one of two ways:
//   * The first tile of a CTA's share is selected exactly. The cutoff comes from
//     group representatives: each thread splits its logits into groups of g and
//     takes one element of each group (the packed signed maximum of its BF16
//     bits, which is the group maximum whenever the group holds a non-negative
//     value). The k-th largest representative, found with a 12-bit histogram,
//     is a lower bound on the tile's k-th largest key, because k distinct
//     elements reach it; and keys above it sit in fewer than about k groups, so
//     they are few. Keys above the cutoff go to a survivor list (one shared
//     atomic per warp); the exact k-th comes from a histogram of survivors
//     relative to the cutoff. When the representatives cannot bound the tile or
//     the survivors overflow, the exact path (g = 1: every key is its own
//     representative) decides it.
//   * Later tiles keep every key at or above a running threshold.
// Either way, a vector is first tested on its packed maximum; the vectors that
// may hold a selected key are queued per warp (ballots), and the warp's lanes
// then work through the queue together, so divergence does not multiply the
// work. Selected keys are appended, in index order, to a candidate buffer at
// slots from warp scans plus one CTA scan of per-run totals: no atomic per key.
// A full buffer is compacted to its exact top-k, which raises the threshold;
// CTAs of a cluster share their lower bounds on the row's k-th key through
// distributed shared memory. The C buffers are merged with cluster-wide
// histograms over distributed shared memory, and each CTA writes its part of
// the answer through the block table, ties at the k-th key split in index order.
// All selection arithmetic is on 16-bit integer keys; no floating point.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "topk_bf16.h"

namespace topk {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int VPT = 8;                       // 16-byte vectors per thread per tile
constexpr int TILE_VEC = THREADS * VPT;      // 2048 vectors = 32 KiB per stage
constexpr int QCAP = 32 * VPT;               // queue entries of one warp
constexpr int HBINS = 4096;                  // 12-bit key bins
constexpr uint32_t SUB_EXACT = 32;           // a bin fuller than this is resolved to the key
constexpr uint32_t KEY_POS_INF = 0xFF80u;    // key of +inf
constexpr uint32_t KEY_NEG_INF = 0x007Fu;    // key of -inf
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // a stage wait gives up after 1 s
constexpr uint32_t NO_ROOM = 0xFFFFFFFFu;

enum : uint32_t { ERR_WAIT = 1u, ERR_BOUNDS = 2u };
enum { CTR_NGT = 0, CTR_NEQ = 1, CTR_SMAX = 2, CTR_BUFMAX = 3 };

__device__ uint32_t g_device_status;

struct Params {
    const uint16_t *logits;
    int64_t row_stride;
    int32_t rows, width;
    const int32_t *valid_len;
    int32_t k;
    const int32_t *table;
    int32_t table_stride, page_shift;
    int32_t *out;
    uint32_t *counters;
    int32_t force_direct;
};

template <int NSTAGE, int CAP, int SURV>
struct alignas(128) Smem {
    uint4 stage[NSTAGE][TILE_VEC];           // streamed logits
    uint32_t buf_idx[CAP];                   // candidate buffer, index order
    uint16_t buf_key[CAP];
    uint16_t surv[SURV];                     // survivors of a tile select
    uint32_t hist[HBINS];                    // 12-bit histogram (zero between uses)
    uint32_t hwin[2][256];                   // window histograms (zero between uses)
    uint32_t h_merge[2][256];                // this CTA's merge histograms (peers read them)
    uint32_t m_all[256];                     // merge: counts over the cluster
    uint32_t m_pre[2][256];                  // merge: counts over lower-ranked CTAs
    uint32_t sub[16];                        // sub-bins of one 12-bit bin
    uint32_t wsum[2][WARPS * VPT];           // run totals, [run * WARPS + warp]
    uint32_t red[2][WARPS];                  // block-scan warp totals
    uint32_t sadj[WARPS][VPT];               // per-run slot offsets of a warp
    uint32_t bc[4];                          // broadcast words
    uint32_t ctr[4];                         // counters (CTR_*)
    uint32_t shared_thr;                     // lower bound on the row's k-th key (max)
    uint32_t shared_max;                     // largest candidate key of the cluster (max)
    uint32_t abort_flag;                     // a bounded wait gave up
    uint8_t queue[WARPS][QCAP];              // per-warp vector queues
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

__device__ __forceinline__ void red_max_peer(uint32_t addr, uint32_t v) {
    asm volatile("red.relaxed.cluster.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(v)
                 : "memory");
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
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
    static constexpr int GMAX = 8;
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

__device__ __forceinline__ int32_t transform(const Params &p, int32_t row, int32_t i) {
    if (!p.table) return i;
    const int32_t page = p.table[static_cast<int64_t>(row) * p.table_stride + (i >> p.page_shift)];
    return (page << p.page_shift) | (i & ((1 << p.page_shift) - 1));
}

// --------------------------------------------------------- the CTA's machinery

template <class M, int NSTAGE, int CAP, int SURV>
struct Cta {
    static constexpr int KPV = M::KPV;
    using S = Smem<NSTAGE, CAP, SURV>;

    S &s;
    const Params &p;
    uint32_t C, rank;
    uint32_t parity = 0;   // alternates double-buffered scan scratch
    // per row
    int32_t row = 0, L = 0;
    int64_t V = 0;
    uint32_t k = 0;
    uint32_t count = 0;    // entries in the candidate buffer
    uint32_t thr = 0;      // keep keys >= thr
    uint32_t buf_lo = 0;   // every buffer key is >= buf_lo
    uint32_t best_T = 0;   // largest exact k-th key found in this CTA's share (0: none)

    __device__ Cta(S &s_, const Params &p_) : s(s_), p(p_) {}

    __device__ __forceinline__ uint32_t effective_thr() {
        if (C > 1) return max(thr, *reinterpret_cast<volatile uint32_t *>(&s.shared_thr));
        return thr;
    }

    // Every CTA of the row learns that the row's k-th key is at least `bound`.
    __device__ __forceinline__ void publish(uint32_t bound) {
        best_T = max(best_T, bound);
        if (C > 1 && threadIdx.x < C && threadIdx.x != rank)
            red_max_peer(peer_addr(&s.shared_thr, threadIdx.x), bound);
    }

    // Inclusive scan over the CTA's threads (one __syncthreads).
    __device__ __forceinline__ uint32_t block_incl_scan(uint32_t x, uint32_t &total) {
        const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
        const uint32_t inc = warp_incl_scan(x);
        if (lane == 31) s.red[parity][warp] = inc;
        __syncthreads();
        const uint32_t w = lane < WARPS ? s.red[parity][lane] : 0u;
        const uint32_t wi = warp_incl_scan(w);
        total = __shfl_sync(0xFFFFFFFFu, wi, 31);
        const uint32_t pre = __shfl_sync(0xFFFFFFFFu, wi - w, warp);
        parity ^= 1u;
        return pre + inc;
    }

    // The 12-bit bin of s.hist holding the q-th largest key: writes s.bc =
    // {bin, above, count(bin)} and returns the histogram total (every thread).
    // Zeroes s.hist. Two __syncthreads.
    __device__ uint32_t find_cut4096(uint32_t q) {
        const int t = threadIdx.x;
        const int base = HBINS - 16 * (t + 1);  // thread 0 owns the highest 16 bins
        uint4 *h4 = reinterpret_cast<uint4 *>(s.hist + base);
        const uint4 a = h4[0], b = h4[1], c = h4[2], d = h4[3];
        const uint32_t v[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w,
                                c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
        const uint4 z = make_uint4(0, 0, 0, 0);
        h4[0] = z;
        h4[1] = z;
        h4[2] = z;
        h4[3] = z;
        uint32_t sum = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) sum += v[i];
        uint32_t total;
        const uint32_t incl = block_incl_scan(sum, total);
        const uint32_t excl = incl - sum;
        if (excl < q && q <= incl) {
            uint32_t acc = excl;
            bool done = false;
#pragma unroll
            for (int i = 15; i >= 0; --i) {
                if (!done && acc + v[i] >= q) {
                    s.bc[0] = static_cast<uint32_t>(base + i);
                    s.bc[1] = acc;
                    s.bc[2] = v[i];
                    done = true;
                }
                acc += v[i];
            }
        }
        __syncthreads();
        return total;
    }

    // The q-th largest of keys[0 .. n), all within [lo, hi] (q <= n): a radix
    // select over bins relative to lo, one pass when hi - lo < 256, else two.
    // T = that key, above = keys greater than it. s.hwin is zero on entry and
    // on exit.
    __device__ void window_select(const uint16_t *keys, uint32_t n, uint32_t lo, uint32_t hi,
                                  uint32_t q, uint32_t &T, uint32_t &above) {
        const int tid = threadIdx.x;
        const uint32_t range = hi - lo;
        const int shift = range < 256u ? 0 : (32 - __clz(static_cast<int>(range))) - 8;
        for (uint32_t i = tid; i < n; i += THREADS)
            atomicAdd(&s.hwin[0][window_bin(keys[i], lo, shift)], 1u);
        __syncthreads();
        uint32_t b1, above1, tot;
        find_bin256(s.hwin[0], q, b1, above1, tot);
        if (shift == 0) {
            T = lo + b1;
            above = above1;
        } else {
            const uint32_t mask = (1u << shift) - 1u;
            for (uint32_t i = tid; i < n; i += THREADS) {
                const uint32_t o = static_cast<uint32_t>(keys[i]) - lo;
                if ((o >> shift) == b1) atomicAdd(&s.hwin[1][o & mask], 1u);
            }
            __syncthreads();
            uint32_t b2, above2;
            find_bin256(s.hwin[1], q - above1, b2, above2, tot);
            T = lo + (b1 << shift) + b2;
            above = above1 + above2;
        }
        __syncthreads();
        s.hwin[0][tid] = 0u;
        s.hwin[1][tid] = 0u;
    }

        // Bin of `key` in a window [lo, lo + (256 << shift)); keys outside it would
    // break the caller's bounds, so they are recorded and clamped.
    __device__ __forceinline__ static uint32_t window_bin(uint32_t key, uint32_t lo, int shift) {
        const uint32_t o = (key - lo) >> shift;
        if (key < lo || o > 255u) {
            atomicOr(&g_device_status, ERR_BOUNDS);
            return key < lo ? 0u : 255u;
        }
        return o;
    }

    // Queue, per warp and in index order, the tile's vectors that may hold a
    // key >= lim. Returns the queue length; run_start[j] = queue position of
    // the first entry of run j (the warp's vectors j*THREADS + warp*32 + lane).
    __device__ __forceinline__ uint32_t build_queue(const uint4 (&raw)[VPT], const uint32_t (&ek)[VPT],
                                                    int nv, uint32_t lim, uint32_t (&run_start)[VPT]) {
        const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
        const uint32_t lt = (1u << lane) - 1u;
        uint32_t q = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int pos = j * THREADS + static_cast<int>(threadIdx.x);
            const bool pass = pos < nv && M::may_reach(raw[j], ek[j], lim);
            const uint32_t b = __ballot_sync(0xFFFFFFFFu, pass);
            run_start[j] = q;
            if (pass) s.queue[warp][q + __popc(b & lt)] = static_cast<uint8_t>((j << 5) | lane);
            q += __popc(b);
        }
        __syncwarp();
        return q;
    }

    // Append to the buffer, in index order, the tile's keys > T and the keys
    // == T while fewer than `take` of them have been taken. Slots: warp scans
    // over the queue plus one CTA scan of the per-run totals. If the result
    // would not fit in `room` slots, nothing is written and NO_ROOM is returned.
    __device__ uint32_t append_pass(const uint4 (&raw)[VPT], const uint32_t (&ek)[VPT],
                                    const uint4 *stg, int64_t tile_v0, int nv, uint32_t T,
                                    uint32_t take, uint32_t room) {
        const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
        uint32_t run_start[VPT];
        const uint32_t Q = build_queue(raw, ek, nv, take ? T : T + 1u, run_start);
        const uint32_t nch = (Q + 31u) >> 5;
        uint32_t pre[VPT];
        uint32_t R[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) R[j] = 0u;
        uint32_t carry = 0, kmax = 0;
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
            pre[m] = 0u;
            if (static_cast<uint32_t>(m) < nch) {
                const uint32_t e = static_cast<uint32_t>(m) * 32u + lane;
                uint32_t cnt = 0, je = VPT;
                if (e < Q) {
                    const uint32_t q = s.queue[warp][e];
                    je = q >> 5;
                    const int pos = static_cast<int>(je) * THREADS + static_cast<int>(warp) * 32 +
                                    static_cast<int>(q & 31u);
                    uint32_t ck[4];
                    M::clean(stg[pos], tile_v0 + pos, V, L, ck);
                    uint32_t gt = 0, eq = 0;
#pragma unroll
                    for (int h = 0; h < KPV; ++h) {
                        const uint32_t key = key_at<M>(ck, h);
                        gt += key > T;
                        eq += key == T;
                        kmax = (key > T || (take && key == T)) ? max(kmax, key) : kmax;
                    }
                    cnt = gt | (eq << 16);
                }
                const uint32_t incl = warp_incl_scan(cnt);
                pre[m] = carry + incl - cnt;
                carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
#pragma unroll
                for (int j = 0; j < VPT; ++j)
                    R[j] += __reduce_add_sync(0xFFFFFFFFu, je == static_cast<uint32_t>(j) ? cnt : 0u);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) s.wsum[parity][j * WARPS + warp] = R[j];
        }
        __syncthreads();
        // Runs in index order: run j of every warp, then run j + 1.
        const uint32_t x0 = s.wsum[parity][lane], x1 = s.wsum[parity][lane + 32];
        const uint32_t s0 = warp_incl_scan(x0);
        const uint32_t t0 = __shfl_sync(0xFFFFFFFFu, s0, 31);
        const uint32_t s1 = warp_incl_scan(x1) + t0;
        const uint32_t total = __shfl_sync(0xFFFFFFFFu, s1, 31);
        const uint32_t ex0 = s0 - x0, ex1 = s1 - x1;
        uint32_t runpre = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const uint32_t f = static_cast<uint32_t>(j) * WARPS + warp;
            const uint32_t base = j < 4 ? __shfl_sync(0xFFFFFFFFu, ex0, f) : __shfl_sync(0xFFFFFFFFu, ex1, f - 32u);
            if (lane == 0) s.sadj[warp][j] = base - runpre;  // packed fields stay non-negative
            runpre += R[j];
        }
        parity ^= 1u;
        const uint32_t gt_total = total & 0xFFFFu, eq_total = total >> 16;
        const uint32_t appended = gt_total + min(eq_total, take);
        if (appended > room) return NO_ROOM;
        kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
        if (lane == 0 && kmax) atomicMax(&s.ctr[CTR_BUFMAX], kmax);
        __syncwarp();
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
            if (static_cast<uint32_t>(m) < nch) {
                const uint32_t e = static_cast<uint32_t>(m) * 32u + lane;
                if (e < Q) {
                    const uint32_t q = s.queue[warp][e];
                    const uint32_t je = q >> 5;
                    const int pos = static_cast<int>(je) * THREADS + static_cast<int>(warp) * 32 +
                                    static_cast<int>(q & 31u);
                    uint32_t ck[4];
                    M::clean(stg[pos], tile_v0 + pos, V, L, ck);
                    const uint32_t off = s.sadj[warp][je] + pre[m];
                    uint32_t gt_before = off & 0xFFFFu, eq_before = off >> 16;
#pragma unroll
                    for (int h = 0; h < KPV; ++h) {
                        const uint32_t key = key_at<M>(ck, h);
                        uint32_t slot = NO_ROOM;
                        if (key > T) {
                            slot = count + gt_before + min(eq_before, take);
                            ++gt_before;
                        } else if (key == T) {
                            if (eq_before < take) slot = count + gt_before + eq_before;
                            ++eq_before;
                        }
                        if (slot != NO_ROOM) {
                            if (slot < static_cast<uint32_t>(CAP)) {
                                s.buf_key[slot] = static_cast<uint16_t>(key);
                                s.buf_idx[slot] = M::elem(tile_v0 + pos, h);
                            } else {
                                atomicOr(&g_device_status, ERR_BOUNDS);
                            }
                        }
                    }
                }
            }
        }
        return appended;
    }

    // Group representatives of this thread's tile, fed to f(key) (0 = none).
    template <int G, class F>
    __device__ __forceinline__ void for_reps(const uint4 (&raw)[VPT], const uint32_t (&ek)[VPT],
                                             int64_t tile_v0, int nv, F &&f) {
        if constexpr (M::BLOCK) {
#pragma unroll
            for (int j = 0; j < VPT; j += G) {
                uint32_t r = 0;
#pragma unroll
                for (int i = 0; i < G; ++i) r = max(r, ek[j + i]);
                f(r >= thr ? r : 0u);
            }
        } else if constexpr (G == 1) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int pos = j * THREADS + static_cast<int>(threadIdx.x);
                uint32_t ck[4] = {0u, 0u, 0u, 0u};
                if (pos < nv) M::clean(raw[j], tile_v0 + pos, V, L, ck);
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const uint32_t key = key_at<M>(ck, h);
                    f(key >= thr ? key : 0u);
                }
            }
        } else if constexpr (G == 2) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                f(rep_key(smax_halves(raw[j].x), thr));
                f(rep_key(smax_halves(raw[j].y), thr));
                f(rep_key(smax_halves(raw[j].z), thr));
                f(rep_key(smax_halves(raw[j].w), thr));
            }
        } else if constexpr (G == 4) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                f(rep_key(smax_halves(smax2(raw[j].x, raw[j].y)), thr));
                f(rep_key(smax_halves(smax2(raw[j].z, raw[j].w)), thr));
            }
        } else {
            constexpr int NV = G / 8;  // vectors per group
#pragma unroll
            for (int j = 0; j < VPT; j += NV) {
                uint32_t m = vec_smax(raw[j]);
#pragma unroll
                for (int i = 1; i < NV; ++i) m = smax2(m, vec_smax(raw[j + i]));
                f(rep_key(smax_halves(m), thr));
            }
        }
    }

    template <int G>
    __device__ __forceinline__ void reps_hist(const uint4 (&raw)[VPT], const uint32_t (&ek)[VPT],
                                              int64_t tile_v0, int nv) {
        for_reps<G>(raw, ek, tile_v0, nv, [&](uint32_t key) {
            if (key) atomicAdd(&s.hist[key >> 4], 1u);
        });
    }

    template <int G>
    __device__ __forceinline__ void reps_sub(const uint4 (&raw)[VPT], const uint32_t (&ek)[VPT],
                                             int64_t tile_v0, int nv, uint32_t bin) {
        for_reps<G>(raw, ek, tile_v0, nv, [&](uint32_t key) {
            if (key && (key >> 4) == bin) atomicAdd(&s.sub[key & 15u], 1u);
        });
    }

    template <class F>
    __device__ __forceinline__ void dispatch_g(int g, F &&f) {
        if constexpr (M::BLOCK) {
            switch (g) {
                case 8: f.template operator()<8>(); break;
                case 4: f.template operator()<4>(); break;
                case 2: f.template operator()<2>(); break;
                default: f.template operator()<1>(); break;
            }
        } else {
            switch (g) {
                case 64: f.template operator()<64>(); break;
                case 32: f.template operator()<32>(); break;
                case 16: f.template operator()<16>(); break;
                case 8: f.template operator()<8>(); break;
                case 4: f.template operator()<4>(); break;
                case 2: f.template operator()<2>(); break;
                default: f.template operator()<1>(); break;
            }
        }
    }

    // Keys > c (and >= thr) of the tile into s.surv (unordered, one shared atomic
    // per warp); keys == c counted; the largest such key. Results in s.ctr after
    // the closing __syncthreads.
    __device__ void survivors(const uint4 (&raw)[VPT], const uint32_t (&ek)[VPT], const uint4 *stg,
                              int64_t tile_v0, int nv, uint32_t c) {
        const uint32_t lane = lane_id(), warp = threadIdx.x >> 5;
        uint32_t run_start[VPT];
        const uint32_t Q = build_queue(raw, ek, nv, max(c, thr), run_start);
        for (uint32_t e0 = 0; e0 < Q; e0 += 32) {
            const uint32_t e = e0 + lane;
            uint32_t ck[4] = {0u, 0u, 0u, 0u};
            if (e < Q) {
                const uint32_t q = s.queue[warp][e];
                const int pos = static_cast<int>(q >> 5) * THREADS + static_cast<int>(warp) * 32 +
                                static_cast<int>(q & 31u);
                M::clean(stg[pos], tile_v0 + pos, V, L, ck);
            }
            uint32_t ngt = 0, neq = 0, kmax = 0;
#pragma unroll
            for (int h = 0; h < KPV; ++h) {
                const uint32_t key = key_at<M>(ck, h);
                const bool ok = key >= thr;
                ngt += ok && key > c;
                neq += ok && key == c;
                kmax = (ok && key > c) ? max(kmax, key) : kmax;
            }
            const uint32_t incl = warp_incl_scan(ngt);
            uint32_t base = 0;
            if (lane == 31 && incl) base = atomicAdd(&s.ctr[CTR_NGT], incl);
            base = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - ngt;
            const uint32_t eqs = __reduce_add_sync(0xFFFFFFFFu, neq);
            const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, kmax);
            if (lane == 0) {
                if (eqs) atomicAdd(&s.ctr[CTR_NEQ], eqs);
                if (mx) atomicMax(&s.ctr[CTR_SMAX], mx);
            }
            if (ngt) {
#pragma unroll
                for (int h = 0; h < KPV; ++h) {
                    const uint32_t key = key_at<M>(ck, h);
                    if (key >= thr && key > c) {
                        if (base < static_cast<uint32_t>(SURV)) s.surv[base] = static_cast<uint16_t>(key);
                        ++base;
                    }
                }
            }
        }
        __syncthreads();
    }

    // Exact top-k of the tile's keys >= thr, appended to the buffer in index
    // order; raises thr when the tile held more than k.
    __device__ void tile_select(const uint4 (&raw)[VPT], const uint32_t (&ek)[VPT], const uint4 *stg,
                                int64_t tile_v0, int nv) {
        const int tid = threadIdx.x;
        const int64_t nE64 = M::BLOCK ? nv
                                      : min(static_cast<int64_t>(nv) * 8, static_cast<int64_t>(L) - 8 * tile_v0);
        const uint32_t nE = static_cast<uint32_t>(nE64);
        uint32_t T = thr - 1u, take = 0;
        bool found = false;
        if (nE <= k) {
            count_event(p, TOPK_CNT_TILE_TAKE_ALL);
        } else {
            // Group size: about 2k representatives (at least k).
            int g = 1;
            if (!p.force_direct) {
                while (g < M::GMAX && nE / static_cast<uint32_t>(2 * g) >= 2u * k) g *= 2;
            } else {
                count_event(p, TOPK_CNT_TILE_FORCED);
            }
            for (;;) {
                if (tid < 4) s.ctr[tid] = tid == CTR_SMAX ? 0u : (tid == CTR_BUFMAX ? s.ctr[tid] : 0u);
                if (tid < 16) s.sub[tid] = 0u;
                dispatch_g(g, [&]<int G>() { reps_hist<G>(raw, ek, tile_v0, nv); });
                __syncthreads();
                const uint32_t NR = find_cut4096(k);
                if (NR < k) {
                    if (g > 1) {  // the representatives cannot bound the tile: exact path
                        count_event(p, TOPK_CNT_TILE_OVERSHOT);
                        g = 1;
                        continue;
                    }
                    count_event(p, TOPK_CNT_TILE_TAKE_ALL);  // at most k candidates
                    break;
                }
                const uint32_t bin = s.bc[0], above = s.bc[1], cnt = s.bc[2];
                uint32_t c, c_above = above;
                if (g == 1 || cnt > SUB_EXACT) {
                    dispatch_g(g, [&]<int G>() { reps_sub<G>(raw, ek, tile_v0, nv, bin); });
                    __syncthreads();
                    uint32_t acc = above, sb = 0;
                    bool done = false;
#pragma unroll
                    for (int i = 15; i >= 0; --i) {
                        const uint32_t v = s.sub[i];
                        if (!done && acc + v >= k) {
                            sb = static_cast<uint32_t>(i);
                            c_above = acc;
                            done = true;
                        }
                        acc += v;
                    }
                    c = (bin << 4) | sb;
                } else {
                    c = max(bin << 4, thr - 1u);  // a lower bound on the k-th representative
                }
                if (g == 1) {
                    // Every key is a representative: c is the k-th key itself.
                    T = c;
                    take = k - c_above;
                    found = true;
                    break;
                }
                survivors(raw, ek, stg, tile_v0, nv, c);
                const uint32_t ngt = s.ctr[CTR_NGT], smax = s.ctr[CTR_SMAX];
                if (ngt > static_cast<uint32_t>(SURV)) {
                    count_event(p, TOPK_CNT_TILE_OVERFLOW);
                    g = 1;
                    __syncthreads();
                    continue;
                }
                count_event(p, TOPK_CNT_TILE_SAMPLED);
                if (ngt >= k) {
                    uint32_t a2;
                    window_select(s.surv, ngt, c + 1u, smax, k, T, a2);
                    take = k - a2;
                } else {
                    T = c;
                    take = k - ngt;
                }
                found = true;
                break;
            }
        }
        const uint32_t room = static_cast<uint32_t>(CAP) - count;
        const uint32_t added = append_pass(raw, ek, stg, tile_v0, nv, T, take, room);
        count += added == NO_ROOM ? 0u : added;
        buf_lo = min(buf_lo, found ? T : thr);
        if (found) {
            // The buffer holds this tile's top-k, all >= T, ahead of any later
            // key: a later key equal to T can no longer be selected.
            thr = max(thr, T + 1u);
            publish(T);
        }
        __syncthreads();
    }

    // Reduce the candidate buffer to its exact top-k, keeping index order.
    __device__ void compact() {
        const int tid = threadIdx.x;
        count_event(p, TOPK_CNT_COMPACTIONS);
        __syncthreads();
        const uint32_t hi = s.ctr[CTR_BUFMAX];
        uint32_t T, above;
        window_select(s.buf_key, count, buf_lo, max(hi, buf_lo), k, T, above);
        const uint32_t take = k - above;
        uint32_t gt_run = 0, eq_run = 0;
        constexpr int PER = 8;
        for (uint32_t base = 0; base < count; base += THREADS * PER) {
            const uint32_t first = base + static_cast<uint32_t>(tid) * PER;
            uint32_t key[PER], idx[PER], gt = 0, eq = 0;
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                const uint32_t i = first + e;
                key[e] = i < count ? s.buf_key[i] : 0u;
                idx[e] = i < count ? s.buf_idx[i] : 0u;
                gt += key[e] > T;
                eq += key[e] == T;
            }
            uint32_t total;
            const uint32_t incl = block_incl_scan(gt | (eq << 16), total);
            const uint32_t ex = incl - (gt | (eq << 16));
            uint32_t gt_before = gt_run + (ex & 0xFFFFu), eq_before = eq_run + (ex >> 16);
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                if (key[e] > T) {
                    const uint32_t slot = gt_before + min(eq_before, take);
                    s.buf_key[slot] = static_cast<uint16_t>(key[e]);
                    s.buf_idx[slot] = idx[e];
                    ++gt_before;
                } else if (key[e] == T) {
                    if (eq_before < take) {
                        const uint32_t slot = gt_before + eq_before;
                        s.buf_key[slot] = static_cast<uint16_t>(key[e]);
                        s.buf_idx[slot] = idx[e];
                    }
                    ++eq_before;
                }
            }
            gt_run += total & 0xFFFFu;
            eq_run += total >> 16;
        }
        count = gt_run + min(eq_run, take);
        buf_lo = T;
        thr = max(thr, T + 1u);
        publish(T);
        __syncthreads();
    }

    // A later tile: append every key >= the threshold.
    __device__ void filter_tile(const uint4 (&raw)[VPT], const uint32_t (&ek)[VPT], const uint4 *stg,
                                int64_t tile_v0, int nv) {
        uint32_t t = effective_thr();
        uint32_t added = append_pass(raw, ek, stg, tile_v0, nv, t - 1u, 0u, static_cast<uint32_t>(CAP) - count);
        if (added == NO_ROOM && count > k) {
            compact();
            t = effective_thr();
            added = append_pass(raw, ek, stg, tile_v0, nv, t - 1u, 0u, static_cast<uint32_t>(CAP) - count);
        }
        if (added == NO_ROOM) {
            // This tile alone holds more than the buffer's room: select its
            // top-k exactly instead.
            count_event(p, TOPK_CNT_OVERFLOW_ROUNDS);
            thr = max(thr, t);
            tile_select(raw, ek, stg, tile_v0, nv);
            return;
        }
        count += added;
        buf_lo = min(buf_lo, t);
    }

    __device__ void emit_single() {
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < k; i += THREADS)
            p.out[static_cast<int64_t>(row) * k + i] =
                i < count ? transform(p, row, static_cast<int32_t>(s.buf_idx[i])) : -1;
    }

    // Cluster merge of the C buffers (each its CTA's top-k, in index order).
    __device__ void merge_and_emit() {
        const int tid = threadIdx.x;
        count_event(p, TOPK_CNT_CLUSTER_MERGES);
        __syncthreads();
        // Every CTA learns the row's best lower bound and its largest key.
        const uint32_t my_max = count ? s.ctr[CTR_BUFMAX] : 0u;
        if (tid == 0) {
            atomicMax(&s.shared_thr, best_T);
            atomicMax(&s.shared_max, my_max);
        }
        if (tid < static_cast<int>(C) && tid != static_cast<int>(rank)) {
            red_max_peer(peer_addr(&s.shared_thr, tid), best_T);
            red_max_peer(peer_addr(&s.shared_max, tid), my_max);
        }
        cluster_arrive();
        cluster_wait();
        const uint32_t LB = max(*reinterpret_cast<volatile uint32_t *>(&s.shared_thr), 1u);
        const uint32_t HI = *reinterpret_cast<volatile uint32_t *>(&s.shared_max);
        const uint32_t range = HI > LB ? HI - LB : 0u;
        const int shift = range < 256u ? 0 : (32 - __clz(static_cast<int>(range))) - 8;
        constexpr int PER = (TOPK_MAX_K + THREADS - 1) / THREADS;
        const uint32_t first = static_cast<uint32_t>(tid) * PER;
        uint32_t key[PER], idx[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const uint32_t i = first + e;
            key[e] = i < count ? s.buf_key[i] : 0u;
            idx[e] = i < count ? s.buf_idx[i] : 0u;
            if (key[e] < LB || HI < LB) key[e] = 0u;  // cannot be selected
            if (key[e]) atomicAdd(&s.h_merge[0][window_bin(key[e], LB, shift)], 1u);
        }
        cluster_arrive();
        cluster_wait();
        {
            uint32_t all = 0, pre = 0;
            for (uint32_t r = 0; r < C; ++r) {
                const uint32_t x = ld_peer(peer_addr(&s.h_merge[0][tid], r));
                all += x;
                pre += r < rank ? x : 0u;
            }
            s.m_all[tid] = all;
            s.m_pre[0][tid] = pre;
        }
        __syncthreads();
        uint32_t b1, above1, total;
        const bool enough = find_bin256(s.m_all, k, b1, above1, total);
        uint32_t T = 0, take = 0, gt_prev = 0, eq_prev = 0, b2 = 0;
        const uint32_t lane = lane_id();
        if (!enough) {
            // Fewer than k candidates in the row: all of them.
            uint32_t x = 0;
            for (uint32_t b = lane; b < 256u; b += 32u) x += s.m_pre[0][b];
            gt_prev = __reduce_add_sync(0xFFFFFFFFu, x);
        } else if (shift == 0) {
            T = LB + b1;
            take = k - above1;
            uint32_t x = 0;
            for (uint32_t b = lane; b < 256u; b += 32u) x += b > b1 ? s.m_pre[0][b] : 0u;
            gt_prev = __reduce_add_sync(0xFFFFFFFFu, x);
            eq_prev = s.m_pre[0][b1];
        } else {
            const uint32_t mask = (1u << shift) - 1u;
#pragma unroll
            for (int e = 0; e < PER; ++e)
                if (key[e] && ((key[e] - LB) >> shift) == b1) atomicAdd(&s.h_merge[1][(key[e] - LB) & mask], 1u);
            __syncthreads();
            cluster_arrive();
            cluster_wait();
            uint32_t all = 0, pre = 0;
            for (uint32_t r = 0; r < C; ++r) {
                const uint32_t x = ld_peer(peer_addr(&s.h_merge[1][tid], r));
                all += x;
                pre += r < rank ? x : 0u;
            }
            s.m_all[tid] = all;
            s.m_pre[1][tid] = pre;
            __syncthreads();
            uint32_t above2, tot2;
            find_bin256(s.m_all, k - above1, b2, above2, tot2);
            T = LB + (b1 << shift) + b2;
            take = k - above1 - above2;
            uint32_t x = 0;
            for (uint32_t b = lane; b < 256u; b += 32u)
                x += (b > b1 ? s.m_pre[0][b] : 0u) + (b > b2 ? s.m_pre[1][b] : 0u);
            gt_prev = __reduce_add_sync(0xFFFFFFFFu, x);
            eq_prev = s.m_pre[1][b2];
        }
        cluster_arrive();  // done reading the peers' shared memory
        // Ordered emission: keys > T, then ties while the row-wide tie rank < take.
        uint32_t gt = 0, eq = 0;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            gt += key[e] != 0u && key[e] > T;
            eq += key[e] != 0u && key[e] == T;
        }
        uint32_t totals;
        const uint32_t incl = block_incl_scan(gt | (eq << 16), totals);
        const uint32_t ex = incl - (gt | (eq << 16));
        const uint32_t quota = take > eq_prev ? take - eq_prev : 0u;
        const uint32_t mine = (totals & 0xFFFFu) + min(totals >> 16, quota);
        const uint32_t offset = gt_prev + min(eq_prev, take);
        uint32_t lgt = ex & 0xFFFFu, leq = ex >> 16;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            if (key[e] == 0u) continue;
            if (key[e] > T) {
                s.buf_idx[lgt + min(leq, quota)] = idx[e];
                ++lgt;
            } else if (key[e] == T) {
                if (leq < quota) s.buf_idx[lgt + leq] = idx[e];
                ++leq;
            }
        }
        __syncthreads();
        const uint32_t selected_total = enough ? k : total;
        int32_t *orow = p.out + static_cast<int64_t>(row) * k;
        for (uint32_t i = tid; i < mine; i += THREADS)
            orow[offset + i] = transform(p, row, static_cast<int32_t>(s.buf_idx[i]));
        for (uint32_t i = selected_total + rank + static_cast<uint32_t>(tid) * C; i < k; i += THREADS * C)
            orow[i] = -1;
        cluster_wait();
        // Every peer is done with this row's shared words: reset them.
        s.h_merge[0][tid] = 0u;
        s.h_merge[1][tid] = 0u;
        if (tid == 0) {
            s.shared_thr = 0u;
            s.shared_max = 0u;
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

template <class M, int NSTAGE, int CAP, int SURV>
__global__ void __launch_bounds__(THREADS, NSTAGE <= 2 ? 2 : 1) topk_kernel(const Params p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    using S = Smem<NSTAGE, CAP, SURV>;
    S &s = *reinterpret_cast<S *>(smem_raw);
    const int tid = threadIdx.x;
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int32_t cid = static_cast<int32_t>(blockIdx.x / C);
    const int32_t ncl = static_cast<int32_t>(gridDim.x / C);

    grid_dependency_wait();
    if (tid == 0) {
        for (int i = 0; i < NSTAGE; ++i) mbar_init(&s.full[i], 1);
        fence_mbar_init();
        s.shared_thr = 0u;
        s.shared_max = 0u;
        s.abort_flag = 0u;
    }
    for (int i = tid; i < HBINS; i += THREADS) s.hist[i] = 0u;
    s.hwin[0][tid] = s.hwin[1][tid] = 0u;
    s.h_merge[0][tid] = s.h_merge[1][tid] = 0u;
    __syncthreads();
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

    Cta<M, NSTAGE, CAP, SURV> cta(s, p);
    cta.C = C;
    cta.rank = rank;
    cta.k = static_cast<uint32_t>(p.k);
    uint32_t seq = 0;
    for (int32_t row = cid; row < p.rows; row += ncl) {
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
        cta.count = 0;
        cta.thr = M::KMIN;
        cta.buf_lo = 0xFFFFu;
        cta.best_T = 0;
        if (tid == 0) s.ctr[CTR_BUFMAX] = 0u;
        const int ntiles = static_cast<int>((v1 - v0 + TILE_VEC - 1) / TILE_VEC);
        for (int i = 0; i < ntiles; ++i, ++seq) {
            const int st = static_cast<int>(seq % NSTAGE);
            const int64_t tile_v0 = v0 + static_cast<int64_t>(i) * TILE_VEC;
            const int nv = static_cast<int>(v1 - tile_v0 < TILE_VEC ? v1 - tile_v0 : TILE_VEC);
            mbar_wait(&s.full[st], (seq / NSTAGE) & 1u, &s.abort_flag);
            count_event(p, TOPK_CNT_ROUNDS);
            const uint4 *stg = s.stage[st];
            uint4 raw[VPT];
            uint32_t ek[VPT];
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int pos = j * THREADS + tid;
                const int64_t v = tile_v0 + pos;
                raw[j] = pos < nv ? stg[pos] : make_uint4(0x80008000u, 0x80008000u, 0x80008000u, 0x80008000u);
                if (!M::BLOCK && pos < nv && v == V - 1 && (L & 7)) {
                    // Lanes past the valid length carry no element.
                    uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
                    const int lanes = L & 7;
#pragma unroll
                    for (int h = 0; h < 8; ++h)
                        if (h >= lanes)
                            w[h >> 1] = (w[h >> 1] & ((h & 1) ? 0x0000FFFFu : 0xFFFF0000u)) |
                                        ((h & 1) ? 0x80000000u : 0x00008000u);
                    raw[j] = make_uint4(w[0], w[1], w[2], w[3]);
                }
                ek[j] = (M::BLOCK && pos < nv) ? BlockMode::key(raw[j], v, V) : 0u;
            }
            if (i == 0) {
                cta.thr = max(cta.thr, cta.effective_thr());
                cta.tile_select(raw, ek, stg, tile_v0, nv);
            } else {
                cta.filter_tile(raw, ek, stg, tile_v0, nv);
            }
            __syncthreads();  // every thread is done with this stage
            if (tid == 0 && feed.row < p.rows) {
                fence_proxy_async();
                feed_issue(feed, s, st, p, M::BLOCK, ncl, C, rank);
            }
        }
        if (cta.count > cta.k) cta.compact();
        if (C == 1) {
            cta.emit_single();
        } else {
            cta.merge_and_emit();
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ host side

struct Variant {
    const void *fn;
    int smem;
};

constexpr int NARROW_NSTAGE = 2, NARROW_CAP = 2048, NARROW_SURV = 4096;
constexpr int WIDE_NSTAGE = 4, WIDE_CAP = 8192, WIDE_SURV = 4096;

template <class M, int NSTAGE, int CAP, int SURV>
Variant variant() {
    return Variant{reinterpret_cast<const void *>(&topk_kernel<M, NSTAGE, CAP, SURV>),
                   static_cast<int>(sizeof(Smem<NSTAGE, CAP, SURV>))};
}

Variant pick(bool block, bool wide) {
    if (block)
        return wide ? variant<BlockMode, WIDE_NSTAGE, WIDE_CAP, WIDE_SURV>()
                    : variant<BlockMode, NARROW_NSTAGE, NARROW_CAP, NARROW_SURV>();
    return wide ? variant<TokenMode, WIDE_NSTAGE, WIDE_CAP, WIDE_SURV>()
                : variant<TokenMode, NARROW_NSTAGE, NARROW_CAP, NARROW_SURV>();
}

struct DeviceInit {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int sms = 0;
    int per_sm[2][2] = {{0, 0}, {0, 0}};   // resident CTAs per SM, [block][wide]
};
DeviceInit g_init[64];

cudaError_t init_device(int dev, DeviceInit *&out) {
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DeviceInit &d = g_init[dev];
    std::call_once(d.once, [&]() {
        cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        for (int b = 0; b < 2 && e == cudaSuccess; ++b)
            for (int w = 0; w < 2 && e == cudaSuccess; ++w) {
                const Variant v = pick(b != 0, w != 0);
                e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem);
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e == cudaSuccess)
                    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.per_sm[b][w], v.fn, THREADS,
                                                                      static_cast<size_t>(v.smem));
                if (e == cudaSuccess && d.per_sm[b][w] < 1) e = cudaErrorInvalidConfiguration;
            }
        d.err = e;
    });
    out = &d;
    return d.err;
}

struct Plan {
    int cluster;
    bool wide;
    int64_t clusters;  // persistent clusters launched
};

// One CTA per row when a row fits one stage. Wider rows: the smallest cluster
// that puts about one CTA on every resident slot, at most 16, and never so many
// CTAs that a share is below one stage. Clusters are persistent, so the grid
// never exceeds what is resident at once.
Plan make_plan(int rows, int width, const DeviceInit &d, bool block, int forced) {
    const int64_t vecs = (static_cast<int64_t>(width) + 7) / 8;
    Plan pl{1, vecs > TILE_VEC, 1};
    if (forced > 0) {
        pl.cluster = forced;
        pl.wide = pl.wide || forced > 1;
    } else if (pl.wide) {
        const int64_t slots = static_cast<int64_t>(d.sms) * d.per_sm[block][1];
        const int64_t stages = (vecs + TILE_VEC - 1) / TILE_VEC;
        int c = 1;
        while (c < 16 && static_cast<int64_t>(rows) * c * 5 < slots * 4 && 2 * c <= stages) c *= 2;
        pl.cluster = c;
    }
    const int64_t slots = static_cast<int64_t>(d.sms) * d.per_sm[block][pl.wide ? 1 : 0];
    const int64_t max_clusters = slots / pl.cluster > 0 ? slots / pl.cluster : 1;
    pl.clusters = rows < max_clusters ? rows : max_clusters;
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
                     int32_t table_stride, int32_t page_size, int32_t *out, void *stream,
                     const topk_bf16_options_t *opt) {
    topk_status_t st = check_args(logits, row_stride, rows, width, valid_len, k, mode, table,
                                  table_stride, page_size, out);
    if (st != TOPK_OK || rows == 0) return st;
    const int forced = opt ? opt->cluster : 0;
    if (forced != 0 && forced != 1 && forced != 2 && forced != 4 && forced != 8 && forced != 16)
        return TOPK_ERR_ARG;
    int dev = 0;
    DeviceInit *d = nullptr;
    if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (init_device(dev, d) != cudaSuccess) return TOPK_ERR_CUDA;

    const bool block = mode == TOPK_BLOCK8;
    const Plan pl = make_plan(rows, width, *d, block, forced);
    const Variant v = pick(block, pl.wide);

    Params prm;
    prm.logits = logits;
    prm.row_stride = row_stride;
    prm.rows = rows;
    prm.width = width;
    prm.valid_len = valid_len;
    prm.k = k;
    prm.table = table;
    prm.table_stride = table_stride;
    prm.page_shift = 0;
    if (table)
        while ((1 << prm.page_shift) < page_size) ++prm.page_shift;
    prm.out = out;
    prm.counters = opt ? opt->counters : nullptr;
    prm.force_direct = opt ? opt->force_direct : 0;

    const int64_t blocks = pl.clusters * pl.cluster;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(v.smem);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(pl.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pl.cluster > 1 ? 1 : 0;  // a lone CTA per row needs no cluster
    void *args[] = {&prm};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, v.fn, args);
    return e == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}

}  // namespace topk

extern "C" {

topk_status_t topk_bf16_select(const uint16_t *logits, int64_t row_stride, int32_t rows,
                               int32_t width, const int32_t *valid_len, int32_t k,
                               topk_mode_t mode, const int32_t *block_table,
                               int32_t table_stride, int32_t page_size, int32_t *out,
                               void *stream) {
    return topk::launch(logits, row_stride, rows, width, valid_len, k, mode, block_table,
                        table_stride, page_size, out, stream, nullptr);
}

topk_status_t topk_bf16_select_ex(const uint16_t *logits, int64_t row_stride, int32_t rows,
                                  int32_t width, const int32_t *valid_len, int32_t k,
                                  topk_mode_t mode, const int32_t *block_table,
                                  int32_t table_stride, int32_t page_size, int32_t *out,
                                  void *stream, const topk_bf16_options_t *options) {
    return topk::launch(logits, row_stride, rows, width, valid_len, k, mode, block_table,
                        table_stride, page_size, out, stream, options);
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
                             int32_t *variant) {
    if (rows < 0 || (mode != TOPK_TOKEN && mode != TOPK_BLOCK8)) return TOPK_ERR_ARG;
    if (k < 1 || k > TOPK_MAX_K) return TOPK_ERR_K;
    if (width < 0 || width > TOPK_MAX_WIDTH) return TOPK_ERR_WIDTH;
    int dev = 0;
    topk::DeviceInit *d = nullptr;
    if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (topk::init_device(dev, d) != cudaSuccess) return TOPK_ERR_CUDA;
    const topk::Plan pl = topk::make_plan(rows, width, *d, mode == TOPK_BLOCK8, 0);
    const topk::Variant v = topk::pick(mode == TOPK_BLOCK8, pl.wide);
    if (cluster) *cluster = pl.cluster;
    if (threads) *threads = topk::THREADS;
    if (smem_bytes) *smem_bytes = v.smem;
    if (variant) *variant = pl.wide ? 1 : 0;
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
