// Exact per-row top-k of BF16 logits for GB300 (sm_103a).
//
// The operation: vLLM "decode_topk_cute", module docstring ("What this module
// computes"); the order key and NaN rule: sglang PR #39305 "Exact bf16 consumer
// top-k adapted from DeepSelect", Modifications; lowest-index ties and the
// block-table transform: vLLM kimi_k3 "dsa/indexer", IndexerSelect.
//
// Design (one cluster of C CTAs per row, C in {1, 2, 4, 8, 16}):
//   * Each CTA owns a contiguous share of the row's valid 16-byte vectors and
//     streams it through a ring of shared-memory stages filled by bulk async
//     copies (cp.async.bulk + mbarrier), one 32 KiB stage per round.
//   * Round 0 of a CTA selects its stage's top-k exactly: a cutoff from one
//     sampled key per vector (a two-pass 8-bit radix select over the samples),
//     then the keys above it (plus at most k ties at it) go to a survivor list
//     whose exact k-th comes from two more 8-bit radix passes. If the sample
//     misjudged the stage (fewer than k keys at or above the cutoff, or too many
//     survivors) the exact path histograms the whole stage instead, with 8
//     replicated copies per CTA so that crowded bins do not serialise.
//   * Later rounds keep only keys at or above a running threshold, tested per
//     vector on its packed maximum first. Selected keys are appended to an
//     index-ordered candidate buffer at slots from a CTA-wide ordered scan (no
//     atomic per key). When the buffer fills, it is compacted to its exact top-k
//     and the threshold rises. CTAs of a cluster share their lower bounds on the
//     row's k-th key through distributed shared memory.
//   * The C buffers are merged with two cluster-wide 8-bit radix histograms over
//     distributed shared memory; each CTA then writes its selected indices, with
//     the ties at the k-th key split in index order across the CTAs.
//   * Indices go out through the block table in one coalesced pass.
// All selection arithmetic is on 16-bit integer keys; no floating point.

#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "topk_bf16.h"

namespace topk {

constexpr int THREADS = 512;
constexpr int WARPS = THREADS / 32;
constexpr int VPT = 4;                       // 16-byte vectors per thread per round
constexpr int STAGE_VEC = THREADS * VPT;     // 2048 vectors = 32 KiB per stage
constexpr int SURV_CAP = 8192;               // survivor keys of a sampled select
constexpr uint32_t KEY_POS_INF = 0xFF80u;    // key of +inf
constexpr uint32_t KEY_NEG_INF = 0x007Fu;    // key of -inf
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // a stage wait gives up after 1 s

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
    int32_t *out;
    uint32_t *counters;
    int32_t force_direct;
};

// ----------------------------------------------------------------- shared memory

template <int NSTAGE, int CAP>
struct alignas(128) Smem {
    uint4 stage[NSTAGE][STAGE_VEC];          // streamed logits
    uint32_t buf_idx[CAP];                   // candidate buffer, index order
    uint16_t buf_key[CAP];
    uint16_t surv[SURV_CAP];                 // survivors of a sampled select
    uint32_t hist_rep[8][256];               // replicated whole-tile histogram
    uint32_t h_samp[2][256];                 // sample select, passes 1 and 2
    uint32_t h_surv[2][256];                 // survivor select
    uint32_t h_full[2][256];                 // whole-tile select (reduced copies)
    uint32_t h_buf[2][256];                  // buffer compaction
    uint32_t h_merge[2][256];                // this CTA's merge histograms (read by peers)
    uint32_t m_all[2][256];                  // merge: sums over the cluster
    uint32_t m_pre[2][256];                  // merge: sums over lower-ranked CTAs
    uint32_t wsum[2][WARPS][4];              // ordered-scan warp totals (double buffered)
    uint32_t ctr[8];
    uint32_t shared_thr;                     // lower bound on the row's k-th key (max)
    uint32_t abort_flag;                     // a bounded wait gave up
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
// raising the CTA's abort flag, which ends every later wait at once). Returns
// whether the phase completed.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity,
                                          volatile uint32_t *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
            *abort = 1u;
            atomicOr(&g_device_status, ERR_WAIT);
            return false;
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

// Mode traits: keys per 16-byte vector, the lowest eligible key, the element
// index of lane h of vector v, and the eligible ("clean") keys of a vector: the
// key where the element may be selected, else 0. Token: NaN and lanes past the
// valid length are ineligible. Block: one key per vector, the NaN-propagating
// maximum of its 8 logits; the newest block is +inf; NaN and -inf blocks are
// ineligible (a selected -inf block would be written as -1, which is what an
// unfilled slot holds anyway).
template <bool BLOCK>
struct Mode;

template <>
struct Mode<false> {
    static constexpr int KPV = 8;
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
    // A superset test: false only if no key of the vector can be >= thr.
    __device__ static __forceinline__ bool may_pass(const uint4 &raw, uint32_t thr) {
        if (thr >= 0x8000u) {
            // Keys >= 0x8000 are exactly the non-negative values, whose keys are
            // their bits + 0x8000: compare the raw bits as signed 16-bit.
            const uint32_t m = __vmaxs2(__vmaxs2(raw.x, raw.y), __vmaxs2(raw.z, raw.w));
            const int32_t a = static_cast<int32_t>(m) >> 16;
            const int32_t b = static_cast<int32_t>(m << 16) >> 16;
            return max(a, b) >= static_cast<int32_t>(thr - 0x8000u);
        }
        const uint32_t m = __vmaxu2(__vmaxu2(key2(raw.x), key2(raw.y)),
                                    __vmaxu2(key2(raw.z), key2(raw.w)));
        return max(m & 0xFFFFu, m >> 16) >= thr;
    }
};

template <>
struct Mode<true> {
    static constexpr int KPV = 1;
    static constexpr uint32_t KMIN = KEY_NEG_INF + 1;
    __device__ static __forceinline__ int32_t elem(int64_t v, int) { return static_cast<int32_t>(v); }
    __device__ static __forceinline__ void clean(const uint4 &raw, int64_t v, int64_t V, int32_t,
                                                 uint32_t (&ck)[4]) {
        uint32_t key;
        if (v == V - 1) {
            key = KEY_POS_INF;  // the newest block is pinned at +inf
        } else if (nan2(raw.x) | nan2(raw.y) | nan2(raw.z) | nan2(raw.w)) {
            key = 0;
        } else {
            const uint32_t m = __vmaxu2(__vmaxu2(key2(raw.x), key2(raw.y)),
                                        __vmaxu2(key2(raw.z), key2(raw.w)));
            key = max(m & 0xFFFFu, m >> 16);
            key = key >= KMIN ? key : 0u;
        }
        ck[0] = key;
        ck[1] = ck[2] = ck[3] = 0;
    }
    __device__ static __forceinline__ bool may_pass(const uint4 &, uint32_t) { return true; }
};

template <bool BLOCK>
__device__ __forceinline__ uint32_t key_at(const uint32_t (&ck)[4], int h) {
    return BLOCK ? ck[0] : (ck[h >> 1] >> ((h & 1) * 16)) & 0xFFFFu;
}

// key_at for a lane chosen at run time, without indexing the register array.
template <bool BLOCK>
__device__ __forceinline__ uint32_t key_at_dyn(const uint32_t (&ck)[4], int h) {
    if (BLOCK) return ck[0];
    const uint32_t w = (h & 4) ? ((h & 2) ? ck[3] : ck[2]) : ((h & 2) ? ck[1] : ck[0]);
    return (w >> ((h & 1) * 16)) & 0xFFFFu;
}

// ------------------------------------------------------------- CTA primitives

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, d);
    return v;
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, d);
        if (lane >= d) v += t;
    }
    return v;
}

// The bin b of a 256-bin histogram (plus `adj` extra counts in bin `adj_bin`)
// holding the q-th largest key: above = count in bins > b, above < q <= above +
// count(b). Run by a whole warp (every warp gets the same answer, so no barrier
// is needed to share it). Returns false when the histogram holds fewer than q.
__device__ __forceinline__ bool find_bin(const uint32_t *hist, uint32_t q, uint32_t adj_bin,
                                         uint32_t adj, uint32_t &bin, uint32_t &above,
                                         uint32_t &total) {
    const int lane = threadIdx.x & 31;
    const int lo_bin = 248 - 8 * lane;  // this lane's bins: lo_bin .. lo_bin + 7
    const uint4 a = *reinterpret_cast<const uint4 *>(hist + lo_bin);
    const uint4 b = *reinterpret_cast<const uint4 *>(hist + lo_bin + 4);
    uint32_t h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] += (static_cast<uint32_t>(lo_bin + i) == adj_bin) ? adj : 0u;
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += h[i];
    const uint32_t incl = warp_incl_scan(s);  // lane 0 holds the highest bins
    total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl >= q);
    if (hit == 0) {
        bin = 0;
        above = total;
        return false;
    }
    const int src = __ffs(hit) - 1;
    uint32_t my_bin = 0, my_above = 0;
    if (lane == src) {
        uint32_t acc = incl - s;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
            if (acc + h[i] >= q) {
                my_bin = lo_bin + i;
                my_above = acc;
                break;
            }
            acc += h[i];
        }
    }
    bin = __shfl_sync(0xFFFFFFFFu, my_bin, src);
    above = __shfl_sync(0xFFFFFFFFu, my_above, src);
    return true;
}

// Exclusive CTA-wide scan of 2*NW 16-bit fields (packed two per word) in
// field-major, thread-minor order. excl[f] = sum of field f over lower threads;
// tot[f] = sum of field f over the CTA. Field totals must stay below 65536.
// Contains one __syncthreads; `parity` alternates the warp-total buffer so that
// consecutive scans need no second barrier.
template <int NW>
__device__ __forceinline__ void ordered_scan(const uint32_t (&v)[NW], uint32_t (&excl)[2 * NW],
                                             uint32_t (&tot)[2 * NW], uint32_t (*wsum)[WARPS][4],
                                             uint32_t &parity) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc[NW];
#pragma unroll
    for (int w = 0; w < NW; ++w) inc[w] = warp_incl_scan(v[w]);
    if (lane == 31) {
#pragma unroll
        for (int w = 0; w < NW; ++w) wsum[parity][warp][w] = inc[w];
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const uint32_t x = lane < WARPS ? wsum[parity][lane][w] : 0u;
        const uint32_t xi = warp_incl_scan(x);
        const uint32_t pre = __shfl_sync(0xFFFFFFFFu, xi - x, warp);
        const uint32_t all = __shfl_sync(0xFFFFFFFFu, xi, 31);
        const uint32_t ex = pre + inc[w] - v[w];
        excl[2 * w] = ex & 0xFFFFu;
        excl[2 * w + 1] = ex >> 16;
        tot[2 * w] = all & 0xFFFFu;
        tot[2 * w + 1] = all >> 16;
    }
    parity ^= 1u;
}

__device__ __forceinline__ void count_event(const Params &p, int which) {
    if (p.counters && threadIdx.x == 0) atomicAdd(p.counters + which, 1u);
}

__device__ __forceinline__ int32_t transform(const Params &p, int32_t row, int32_t i) {
    if (!p.table) return i;
    const int32_t page = p.table[static_cast<int64_t>(row) * p.table_stride + (i >> p.page_shift)];
    return (page << p.page_shift) | (i & ((1 << p.page_shift) - 1));
}

// ------------------------------------------------------------ the CTA's state

template <bool BLOCK, int NSTAGE, int CAP>
struct Cta {
    using M = Mode<BLOCK>;
    using S = Smem<NSTAGE, CAP>;
    static constexpr int KPV = M::KPV;

    S &s;
    const Params &p;
    int32_t row, L, k;
    int64_t V;           // valid vectors of the row
    uint32_t C, rank;
    uint32_t count = 0;  // entries in the candidate buffer
    uint32_t thr;        // keep keys >= thr
    uint32_t parity = 0;

    __device__ Cta(S &s_, const Params &p_) : s(s_), p(p_) {}

    __device__ __forceinline__ uint32_t effective_thr() {
        if (C > 1) {
            const uint32_t shared = *reinterpret_cast<volatile uint32_t *>(&s.shared_thr);
            return max(thr, shared);
        }
        return thr;
    }

    // Tell the other CTAs of the row that its k-th key is at least `bound`.
    __device__ __forceinline__ void publish(uint32_t bound) {
        if (C > 1 && threadIdx.x < C && threadIdx.x != rank)
            red_max_peer(peer_addr(&s.shared_thr, threadIdx.x), bound);
    }

    // Append the selected keys of a register tile: keys > T, and keys == T while
    // fewer than `take` ties have been taken (in index order), at buffer slots
    // from an ordered scan. Returns the number appended.
    __device__ uint32_t append_selected(const uint32_t (&ck)[VPT][4], const int64_t (&vec)[VPT],
                                        uint32_t T, uint32_t take) {
        uint32_t cnt[VPT];  // gt in the low half, eq in the high half
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            uint32_t gt = 0, eq = 0;
#pragma unroll
            for (int h = 0; h < KPV; ++h) {
                const uint32_t key = key_at<BLOCK>(ck[j], h);
                gt += key > T;
                eq += key == T;
            }
            cnt[j] = gt | (eq << 16);
        }
        uint32_t excl[2 * VPT], tot[2 * VPT];
        ordered_scan<VPT>(cnt, excl, tot, s.wsum, parity);
        uint32_t gt_total = 0, eq_total = 0;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            uint32_t gt_before = gt_total + excl[2 * j];
            uint32_t eq_before = eq_total + excl[2 * j + 1];
            gt_total += tot[2 * j];
            eq_total += tot[2 * j + 1];
            if (cnt[j] == 0) continue;
#pragma unroll
            for (int h = 0; h < KPV; ++h) {
                const uint32_t key = key_at<BLOCK>(ck[j], h);
                if (key > T) {
                    const uint32_t slot = count + gt_before + min(eq_before, take);
                    if (slot < CAP) {
                        s.buf_key[slot] = static_cast<uint16_t>(key);
                        s.buf_idx[slot] = M::elem(vec[j], h);
                    } else {
                        atomicOr(&g_device_status, ERR_BOUNDS);
                    }
                    ++gt_before;
                } else if (key == T) {
                    if (eq_before < take) {
                        const uint32_t slot = count + gt_before + eq_before;
                        if (slot < CAP) {
                            s.buf_key[slot] = static_cast<uint16_t>(key);
                            s.buf_idx[slot] = M::elem(vec[j], h);
                        } else {
                            atomicOr(&g_device_status, ERR_BOUNDS);
                        }
                    }
                    ++eq_before;
                }
            }
        }
        return gt_total + min(eq_total, take);
    }

    // Exact top-k of the register tile's keys >= thr, appended to the buffer.
    // ck: clean keys (0 = ineligible); keys below thr are zeroed here.
    __device__ void tile_select(uint32_t (&ck)[VPT][4], const int64_t (&vec)[VPT]) {
        const int tid = threadIdx.x, lane = tid & 31;
        const uint32_t kk = static_cast<uint32_t>(k);
        uint32_t ncand = 0, nsamp = 0;
        uint32_t samp[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                uint32_t lo = ck[j][w] & 0xFFFFu, hi = ck[j][w] >> 16;
                lo = lo >= thr ? lo : 0u;
                hi = hi >= thr ? hi : 0u;
                ck[j][w] = lo | (hi << 16);
                ncand += (lo != 0) + (hi != 0);
            }
            const int pos = j * THREADS + tid;
            samp[j] = key_at_dyn<BLOCK>(ck[j], (pos ^ (pos >> 3)) & 7);
            nsamp += samp[j] != 0;
        }
        // Zero the histograms of this select and the counters.
        for (int i = tid; i < 256; i += THREADS) {
            s.h_samp[0][i] = s.h_samp[1][i] = 0;
            s.h_surv[0][i] = s.h_surv[1][i] = 0;
        }
        if (tid < 8) s.ctr[tid] = 0;
        __syncthreads();
        {
            const uint32_t a = warp_sum(ncand), b = warp_sum(nsamp);
            if (lane == 0) {
                atomicAdd(&s.ctr[0], a);
                atomicAdd(&s.ctr[1], b);
            }
        }
        __syncthreads();
        const uint32_t NC = s.ctr[0], NS = s.ctr[1];
        uint32_t T, take;
        if (NC <= kk) {
            // Every candidate is selected.
            count_event(p, TOPK_CNT_TILE_TAKE_ALL);
            T = thr - 1;
            take = 0;
        } else {
            bool direct = p.force_direct != 0;
            if (direct) count_event(p, TOPK_CNT_TILE_FORCED);
            if (!direct) {
                // Cutoff c: the q-th largest sampled key, q aiming at about 2k
                // survivors (c = thr when the sample is too small to help).
                const uint64_t q64 = (2ull * kk * NS) / NC;
                const uint32_t q = q64 < 1 ? 1u : static_cast<uint32_t>(q64);
                uint32_t c = thr;
                if (q < NS) {
#pragma unroll
                    for (int j = 0; j < VPT; ++j)
                        if (samp[j]) atomicAdd(&s.h_samp[0][samp[j] >> 8], 1u);
                    __syncthreads();
                    uint32_t b1, above1, tot;
                    find_bin(s.h_samp[0], q, 0, 0, b1, above1, tot);
#pragma unroll
                    for (int j = 0; j < VPT; ++j)
                        if (samp[j] && (samp[j] >> 8) == b1) atomicAdd(&s.h_samp[1][samp[j] & 0xFFu], 1u);
                    __syncthreads();
                    uint32_t b2, above2;
                    find_bin(s.h_samp[1], q - above1, 0, 0, b2, above2, tot);
                    c = max(thr, (b1 << 8) | b2);
                }
                // Survivors: keys > c into the list (one shared atomic per warp),
                // ties at c only counted; their high bytes histogrammed on the way.
                uint32_t ngt = 0, neq = 0;
#pragma unroll
                for (int j = 0; j < VPT; ++j)
#pragma unroll
                    for (int h = 0; h < KPV; ++h) {
                        const uint32_t key = key_at<BLOCK>(ck[j], h);
                        ngt += key > c;
                        neq += key == c;
                    }
                const uint32_t incl = warp_incl_scan(ngt);
                uint32_t base = 0;
                if (lane == 31) base = atomicAdd(&s.ctr[2], incl);
                base = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - ngt;
                {
                    const uint32_t e = warp_sum(neq);
                    if (lane == 0 && e) atomicAdd(&s.ctr[3], e);
                }
                if (ngt) {
#pragma unroll
                    for (int j = 0; j < VPT; ++j)
#pragma unroll
                        for (int h = 0; h < KPV; ++h) {
                            const uint32_t key = key_at<BLOCK>(ck[j], h);
                            if (key > c) {
                                if (base < SURV_CAP) {
                                    s.surv[base] = static_cast<uint16_t>(key);
                                    atomicAdd(&s.h_surv[0][key >> 8], 1u);
                                }
                                ++base;
                            }
                        }
                }
                __syncthreads();
                const uint32_t NGT = s.ctr[2], NEQ = s.ctr[3];
                if (NGT + NEQ < kk) {
                    direct = true;  // the cutoff was above the k-th key
                    count_event(p, TOPK_CNT_TILE_OVERSHOT);
                } else if (NGT > SURV_CAP) {
                    direct = true;  // too many survivors to hold
                    count_event(p, TOPK_CNT_TILE_OVERFLOW);
                } else {
                    count_event(p, TOPK_CNT_TILE_SAMPLED);
                    const uint32_t ties = min(NEQ, kk);
                    uint32_t b1, above1, tot;
                    find_bin(s.h_surv[0], kk, c >> 8, ties, b1, above1, tot);
                    for (uint32_t i = tid; i < NGT; i += THREADS) {
                        const uint32_t key = s.surv[i];
                        if ((key >> 8) == b1) atomicAdd(&s.h_surv[1][key & 0xFFu], 1u);
                    }
                    __syncthreads();
                    uint32_t b2, above2;
                    find_bin(s.h_surv[1], kk - above1, c & 0xFFu, (c >> 8) == b1 ? ties : 0u, b2,
                             above2, tot);
                    T = (b1 << 8) | b2;
                    take = kk - above1 - above2;
                }
            }
            if (direct) {
                // Exact path over the whole tile: 8 copies of each histogram,
                // lane l counting into copy l % 8.
                const int copy = lane & 7;
                for (int i = tid; i < 8 * 256; i += THREADS) (&s.hist_rep[0][0])[i] = 0;
                __syncthreads();
#pragma unroll
                for (int j = 0; j < VPT; ++j)
#pragma unroll
                    for (int h = 0; h < KPV; ++h) {
                        const uint32_t key = key_at<BLOCK>(ck[j], h);
                        if (key) atomicAdd(&s.hist_rep[copy][key >> 8], 1u);
                    }
                __syncthreads();
                for (int b = tid; b < 256; b += THREADS) {
                    uint32_t sum = 0;
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        sum += s.hist_rep[r][b];
                        s.hist_rep[r][b] = 0;
                    }
                    s.h_full[0][b] = sum;
                }
                __syncthreads();
                uint32_t b1, above1, tot;
                find_bin(s.h_full[0], kk, 0, 0, b1, above1, tot);
#pragma unroll
                for (int j = 0; j < VPT; ++j)
#pragma unroll
                    for (int h = 0; h < KPV; ++h) {
                        const uint32_t key = key_at<BLOCK>(ck[j], h);
                        if (key && (key >> 8) == b1) atomicAdd(&s.hist_rep[copy][key & 0xFFu], 1u);
                    }
                __syncthreads();
                for (int b = tid; b < 256; b += THREADS) {
                    uint32_t sum = 0;
#pragma unroll
                    for (int r = 0; r < 8; ++r) sum += s.hist_rep[r][b];
                    s.h_full[1][b] = sum;
                }
                __syncthreads();
                uint32_t b2, above2;
                find_bin(s.h_full[1], kk - above1, 0, 0, b2, above2, tot);
                T = (b1 << 8) | b2;
                take = kk - above1 - above2;
            }
        }
        const uint32_t added = append_selected(ck, vec, T, take);
        count += added;
        if (NC > kk) {
            // The buffer now holds this tile's top-k, all at or above T, in index
            // order: a later key equal to T can no longer be selected.
            thr = max(thr, T + 1);
            publish(T);
        }
        __syncthreads();
    }

    // Reduce the candidate buffer to its exact top-k (index order kept).
    __device__ void compact() {
        const int tid = threadIdx.x;
        const uint32_t kk = static_cast<uint32_t>(k);
        count_event(p, TOPK_CNT_COMPACTIONS);
        for (int i = tid; i < 256; i += THREADS) s.h_buf[0][i] = s.h_buf[1][i] = 0;
        __syncthreads();
        constexpr int PER = CAP / THREADS;
        const uint32_t first = tid * PER;
        uint32_t key[PER], idx[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const uint32_t i = first + e;
            key[e] = i < count ? s.buf_key[i] : 0u;
            idx[e] = i < count ? s.buf_idx[i] : 0u;
            if (key[e]) atomicAdd(&s.h_buf[0][key[e] >> 8], 1u);
        }
        __syncthreads();
        uint32_t b1, above1, tot;
        find_bin(s.h_buf[0], kk, 0, 0, b1, above1, tot);
#pragma unroll
        for (int e = 0; e < PER; ++e)
            if (key[e] && (key[e] >> 8) == b1) atomicAdd(&s.h_buf[1][key[e] & 0xFFu], 1u);
        __syncthreads();
        uint32_t b2, above2;
        find_bin(s.h_buf[1], kk - above1, 0, 0, b2, above2, tot);
        const uint32_t T = (b1 << 8) | b2, take = kk - above1 - above2;
        uint32_t gt = 0, eq = 0;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            gt += key[e] > T;
            eq += key[e] == T;
        }
        uint32_t v[1] = {gt | (eq << 16)}, excl[2], totals[2];
        ordered_scan<1>(v, excl, totals, s.wsum, parity);  // all reads done before it
        uint32_t gt_before = excl[0], eq_before = excl[1];
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
        count = totals[0] + min(totals[1], take);  // == k
        thr = max(thr, T + 1);
        publish(T);
        __syncthreads();
    }

    // A later round: append every key >= the threshold.
    __device__ void filter_round(const uint4 (&raw)[VPT], const int64_t (&vec)[VPT],
                                 const bool (&valid)[VPT]) {
        uint32_t t = effective_thr();
        uint32_t ck[VPT][4];
        uint32_t cnt[VPT];
        for (int attempt = 0;; ++attempt) {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                cnt[j] = 0;
                ck[j][0] = ck[j][1] = ck[j][2] = ck[j][3] = 0;
                if (valid[j] && M::may_pass(raw[j], t)) {
                    M::clean(raw[j], vec[j], V, L, ck[j]);
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t lo = ck[j][w] & 0xFFFFu, hi = ck[j][w] >> 16;
                        lo = lo >= t ? lo : 0u;
                        hi = hi >= t ? hi : 0u;
                        ck[j][w] = lo | (hi << 16);
                        cnt[j] += (lo != 0) + (hi != 0);
                    }
                }
            }
            uint32_t v[VPT / 2], excl[VPT], tot[VPT];
#pragma unroll
            for (int w = 0; w < VPT / 2; ++w) v[w] = cnt[2 * w] | (cnt[2 * w + 1] << 16);
            ordered_scan<VPT / 2>(v, excl, tot, s.wsum, parity);
            uint32_t total = 0;
#pragma unroll
            for (int j = 0; j < VPT; ++j) total += tot[j];
            if (count + total <= static_cast<uint32_t>(CAP)) {
                uint32_t base = count;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    uint32_t slot = base + excl[j];
                    base += tot[j];
                    if (cnt[j] == 0) continue;
#pragma unroll
                    for (int h = 0; h < KPV; ++h) {
                        const uint32_t key = key_at<BLOCK>(ck[j], h);
                        if (key) {
                            s.buf_key[slot] = static_cast<uint16_t>(key);
                            s.buf_idx[slot] = M::elem(vec[j], h);
                            ++slot;
                        }
                    }
                }
                count += total;
                return;
            }
            // The buffer would overflow: compact it (raising the threshold) and
            // count again; if the round alone is still too large, select its
            // top-k exactly instead.
            if (attempt == 0 && count > static_cast<uint32_t>(k)) {
                compact();
                t = effective_thr();
                continue;
            }
            count_event(p, TOPK_CNT_OVERFLOW_ROUNDS);
            if (count > static_cast<uint32_t>(k)) compact();
            thr = max(thr, effective_thr());
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                ck[j][0] = ck[j][1] = ck[j][2] = ck[j][3] = 0;
                if (valid[j]) M::clean(raw[j], vec[j], V, L, ck[j]);
            }
            tile_select(ck, vec);
            return;
        }
    }

    // Write this CTA's buffer (C == 1: the row's answer) through the table.
    __device__ void emit_single() {
        for (int sidx = threadIdx.x; sidx < k; sidx += THREADS)
            p.out[static_cast<int64_t>(row) * k + sidx] =
                sidx < static_cast<int>(count) ? transform(p, row, static_cast<int32_t>(s.buf_idx[sidx]))
                                               : -1;
    }

    // Cluster merge of the C buffers (each already its CTA's top-k, index order).
    __device__ void merge_and_emit() {
        const int tid = threadIdx.x;
        const uint32_t kk = static_cast<uint32_t>(k);
        count_event(p, TOPK_CNT_CLUSTER_MERGES);
        constexpr int PER = (TOPK_MAX_K + THREADS - 1) / THREADS;  // count <= k entries
        const uint32_t first = tid * PER;
        uint32_t key[PER], idx[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const uint32_t i = first + e;
            key[e] = i < count ? s.buf_key[i] : 0u;
            idx[e] = i < count ? s.buf_idx[i] : 0u;
            if (key[e]) atomicAdd(&s.h_merge[0][key[e] >> 8], 1u);
        }
        cluster_arrive();
        cluster_wait();
        for (int b = tid; b < 256; b += THREADS) {
            uint32_t all = 0, pre = 0;
            for (uint32_t r = 0; r < C; ++r) {
                const uint32_t x = ld_peer(peer_addr(&s.h_merge[0][b], r));
                all += x;
                pre += r < rank ? x : 0u;
            }
            s.m_all[0][b] = all;
            s.m_pre[0][b] = pre;
        }
        __syncthreads();
        uint32_t b1, above1, total;
        const bool enough = find_bin(s.m_all[0], kk, 0, 0, b1, above1, total);
        uint32_t T, take, gt_prev, eq_prev;
        const int lane = tid & 31;
        if (!enough) {
            // Fewer than k candidates in the whole row: take them all.
            T = 0;
            take = 0;
            uint32_t x = 0;
            for (int b = lane; b < 256; b += 32) x += s.m_pre[0][b];
            gt_prev = warp_sum(x);
            eq_prev = 0;
        } else {
#pragma unroll
            for (int e = 0; e < PER; ++e)
                if (key[e] && (key[e] >> 8) == b1) atomicAdd(&s.h_merge[1][key[e] & 0xFFu], 1u);
            cluster_arrive();
            cluster_wait();
            for (int b = tid; b < 256; b += THREADS) {
                uint32_t all = 0, pre = 0;
                for (uint32_t r = 0; r < C; ++r) {
                    const uint32_t x = ld_peer(peer_addr(&s.h_merge[1][b], r));
                    all += x;
                    pre += r < rank ? x : 0u;
                }
                s.m_all[1][b] = all;
                s.m_pre[1][b] = pre;
            }
            __syncthreads();
            uint32_t b2, above2, tot2;
            find_bin(s.m_all[1], kk - above1, 0, 0, b2, above2, tot2);
            T = (b1 << 8) | b2;
            take = kk - above1 - above2;
            uint32_t x = 0;
            for (int b = lane; b < 256; b += 32)
                x += (static_cast<uint32_t>(b) > b1 ? s.m_pre[0][b] : 0u) +
                     (static_cast<uint32_t>(b) > b2 ? s.m_pre[1][b] : 0u);
            gt_prev = warp_sum(x);
            eq_prev = s.m_pre[1][b2];
        }
        cluster_arrive();  // done reading the peers' shared memory
        // Ordered emission: keys > T, and ties while the row-wide tie rank < take.
        // Ties in lower-ranked CTAs come first, so this CTA may take `quota`.
        uint32_t gt = 0, eq = 0;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            gt += key[e] != 0 && key[e] > T;
            eq += key[e] != 0 && key[e] == T;
        }
        uint32_t v[1] = {gt | (eq << 16)}, excl[2], totals[2];
        ordered_scan<1>(v, excl, totals, s.wsum, parity);  // all buffer reads happened above
        const uint32_t quota = take > eq_prev ? take - eq_prev : 0u;
        const uint32_t mine = totals[0] + min(totals[1], quota);
        const uint32_t offset = gt_prev + min(eq_prev, take);
        uint32_t lgt = excl[0], leq = excl[1];
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            if (key[e] == 0) continue;
            if (key[e] > T) {
                s.buf_idx[lgt + min(leq, quota)] = idx[e];
                ++lgt;
            } else if (key[e] == T) {
                if (leq < quota) s.buf_idx[lgt + leq] = idx[e];
                ++leq;
            }
        }
        __syncthreads();
        const uint32_t selected_total = enough ? kk : total;
        for (uint32_t i = tid; i < mine; i += THREADS)
            p.out[static_cast<int64_t>(row) * k + offset + i] =
                transform(p, row, static_cast<int32_t>(s.buf_idx[i]));
        for (uint32_t i = selected_total + rank + tid * C; i < kk; i += THREADS * C)
            p.out[static_cast<int64_t>(row) * k + i] = -1;
        cluster_wait();
    }
};

template <bool BLOCK, int NSTAGE, int CAP>
__global__ void __launch_bounds__(THREADS, 1) topk_kernel(const Params p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    using S = Smem<NSTAGE, CAP>;
    S &s = *reinterpret_cast<S *>(smem_raw);
    const int tid = threadIdx.x;
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int32_t row = static_cast<int32_t>(blockIdx.x / C);
    if (row >= p.rows) return;

    grid_dependency_wait();
    const int32_t L = min(max(__ldg(p.valid_len + row), 0), p.width);
    const int32_t n = BLOCK ? (L + 7) >> 3 : L;
    if (n <= p.k) {
        // At most k elements: 0 .. n-1, then -1, without reading the logits.
        if (rank == 0) count_event(p, TOPK_CNT_BYPASS_ROWS);
        const int32_t lo = static_cast<int32_t>(static_cast<int64_t>(p.k) * rank / C);
        const int32_t hi = static_cast<int32_t>(static_cast<int64_t>(p.k) * (rank + 1) / C);
        for (int32_t i = lo + tid; i < hi; i += THREADS)
            p.out[static_cast<int64_t>(row) * p.k + i] = i < n ? transform(p, row, i) : -1;
        return;
    }

    Cta<BLOCK, NSTAGE, CAP> cta(s, p);
    cta.row = row;
    cta.L = L;
    cta.k = p.k;
    cta.V = (static_cast<int64_t>(L) + 7) >> 3;
    cta.C = C;
    cta.rank = rank;
    cta.thr = Mode<BLOCK>::KMIN;

    const int64_t v0 = cta.V * rank / C, v1 = cta.V * (rank + 1) / C;
    const int64_t nvec = v1 - v0;
    const int rounds = static_cast<int>((nvec + STAGE_VEC - 1) / STAGE_VEC);
    const uint4 *src = reinterpret_cast<const uint4 *>(p.logits + static_cast<int64_t>(row) * p.row_stride);

    if (tid == 0) {
        for (int i = 0; i < NSTAGE; ++i) mbar_init(&s.full[i], 1);
        fence_mbar_init();
    }
    for (int i = tid; i < 2 * 256; i += THREADS) (&s.h_merge[0][0])[i] = 0;
    if (tid == 0) {
        s.shared_thr = 0;
        s.abort_flag = 0;
    }
    __syncthreads();
    if (tid == 0) {
        for (int i = 0; i < NSTAGE && i < rounds; ++i) {
            const int64_t b = v0 + static_cast<int64_t>(i) * STAGE_VEC;
            const uint32_t bytes = static_cast<uint32_t>((v1 - b < STAGE_VEC ? v1 - b : STAGE_VEC) * 16);
            mbar_expect_tx(&s.full[i], bytes);
            bulk_load(&s.stage[i][0], src + b, bytes, &s.full[i]);
        }
    }
    if (C > 1) {
        // Every CTA of the cluster has started and zeroed its shared words
        // before any distributed shared memory access.
        cluster_arrive();
        cluster_wait();
    }

    for (int i = 0; i < rounds; ++i) {
        const int st = i % NSTAGE;
        const int64_t base = v0 + static_cast<int64_t>(i) * STAGE_VEC;
        const int64_t nv = v1 - base < STAGE_VEC ? v1 - base : STAGE_VEC;
        mbar_wait(&s.full[st], static_cast<uint32_t>(i / NSTAGE) & 1u, &s.abort_flag);
        count_event(p, TOPK_CNT_ROUNDS);
        uint4 raw[VPT];
        int64_t vec[VPT];
        bool valid[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int pos = j * THREADS + tid;
            valid[j] = pos < nv;
            vec[j] = base + pos;
            raw[j] = valid[j] ? s.stage[st][pos] : make_uint4(0, 0, 0, 0);
        }
        if (i == 0) {
            uint32_t ck[VPT][4];
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                ck[j][0] = ck[j][1] = ck[j][2] = ck[j][3] = 0;
                if (valid[j]) Mode<BLOCK>::clean(raw[j], vec[j], cta.V, L, ck[j]);
            }
            cta.thr = max(cta.thr, cta.effective_thr());
            cta.tile_select(ck, vec);
        } else {
            cta.filter_round(raw, vec, valid);
        }
        __syncthreads();  // every thread is done with this stage
        if (tid == 0 && i + NSTAGE < rounds) {
            const int64_t b = v0 + static_cast<int64_t>(i + NSTAGE) * STAGE_VEC;
            const uint32_t bytes = static_cast<uint32_t>((v1 - b < STAGE_VEC ? v1 - b : STAGE_VEC) * 16);
            fence_proxy_async();
            mbar_expect_tx(&s.full[st], bytes);
            bulk_load(&s.stage[st][0], src + b, bytes, &s.full[st]);
        }
    }
    if (cta.count > static_cast<uint32_t>(p.k)) cta.compact();
    if (C == 1) {
        cta.emit_single();
    } else {
        cta.merge_and_emit();
    }
}

// ------------------------------------------------------------------ host side

struct Variant {
    const void *fn;
    int smem;
};

template <bool BLOCK, int NSTAGE, int CAP>
Variant variant() {
    return Variant{reinterpret_cast<const void *>(&topk_kernel<BLOCK, NSTAGE, CAP>),
                   static_cast<int>(sizeof(Smem<NSTAGE, CAP>))};
}

constexpr int NARROW_NSTAGE = 1, NARROW_CAP = 2048;
constexpr int WIDE_NSTAGE = 3, WIDE_CAP = 8192;

Variant pick(bool block, bool wide) {
    if (block) return wide ? variant<true, WIDE_NSTAGE, WIDE_CAP>() : variant<true, NARROW_NSTAGE, NARROW_CAP>();
    return wide ? variant<false, WIDE_NSTAGE, WIDE_CAP>() : variant<false, NARROW_NSTAGE, NARROW_CAP>();
}

struct DeviceInit {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int sms = 0;
};
DeviceInit g_init[64];

cudaError_t init_device(int dev, int &sms) {
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
            }
        d.err = e;
    });
    sms = d.sms;
    return d.err;
}

struct Plan {
    int cluster;
    bool wide;
};

// CTAs per row: one for rows that fit a stage; otherwise enough to keep about
// two CTAs' worth of rows per SM in flight, at most 16 and never so many that a
// CTA's share is below one stage.
Plan make_plan(int rows, int width, bool block, int sms, int forced) {
    const int64_t vecs = (static_cast<int64_t>(width) + 7) / 8;
    Plan pl{1, vecs > STAGE_VEC};
    if (forced > 0) {
        pl.cluster = forced;
        pl.wide = pl.wide || forced > 1;
        return pl;
    }
    if (!pl.wide) return pl;
    int c = 1;
    const int64_t stages = (vecs + STAGE_VEC - 1) / STAGE_VEC;
    while (c < 16 && static_cast<int64_t>(rows) * c * 2 <= 2LL * sms && 2 * c <= stages) c *= 2;
    pl.cluster = c;
    (void)block;
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
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (init_device(dev, sms) != cudaSuccess) return TOPK_ERR_CUDA;

    const bool block = mode == TOPK_BLOCK8;
    const Plan pl = make_plan(rows, width, block, sms, forced);
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

    const int64_t blocks = static_cast<int64_t>(rows) * pl.cluster;
    if (blocks > 0x7FFFFFFF) return TOPK_ERR_ARG;
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
    cfg.numAttrs = 1;
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
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (topk::init_device(dev, sms) != cudaSuccess) return TOPK_ERR_CUDA;
    const topk::Plan pl = topk::make_plan(rows, width, mode == TOPK_BLOCK8, sms, 0);
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
