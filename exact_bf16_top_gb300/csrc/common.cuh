// Device building blocks shared by the library's kernels: bulk copies and
// mbarriers, cluster and distributed-shared-memory access, programmatic
// dependent launch, the order-preserving 16-bit keys, warp scans, histogram
// searches and the block-table transform.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "params.h"
#include "topk_bf16.h"

namespace topk {

// The device-side error word (a bounded wait that gave up, a failed internal
// capacity check): one per translation unit, read by the host through the
// unit's status function. Kernels never trap.
static __device__ uint32_t g_device_status;

// Debug builds (-DTOPK_DEBUG): every shared-memory index a kernel computes from
// data (a count, a scan, an atomic's result, a key) is checked before use with
// TOPK_IDX_OK(i, n); an index outside [0, n) sets ERR_DEBUG_INDEX in the status
// word and the access is skipped (no trap). Release builds compile the checks
// away.
#ifdef TOPK_DEBUG
__device__ __forceinline__ bool debug_index_ok(uint64_t i, uint64_t n) {
    if (i < n) return true;
    atomicOr(&g_device_status, ERR_DEBUG_INDEX);
    return false;
}
#define TOPK_IDX_OK(i, n) ::topk::debug_index_ok(static_cast<uint64_t>(i), static_cast<uint64_t>(n))
#else
#define TOPK_IDX_OK(i, n) true
#endif

static cudaError_t unit_status(uint32_t *v, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_device_status, sizeof(uint32_t));
    if (e == cudaSuccess && clear) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
    }
    return e;
}

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

// As mbar_try_wait, but a thread whose phase is not complete yet may be
// suspended for up to `hint_ns` (it resumes as soon as the phase completes), so
// that a waiting CTA issues few instructions while others on the SM work.
__device__ __forceinline__ bool mbar_try_wait_hint(unsigned long long *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
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

// mbar_wait for a CTA that shares its SM with others: each try may suspend
// the waiting threads (up to 20 us, resumed at the phase's completion) instead
// of spinning; the same 1 s limit.
__device__ __forceinline__ void mbar_wait_sleep(unsigned long long *bar, uint32_t parity,
                                                volatile uint32_t *abort) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_hint(bar, parity, 20000u)) return;
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

__device__ __forceinline__ void red_add_peer(uint32_t addr, uint32_t v) {
    asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v)
                 : "memory");
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

// ---------------------------------------------------------- packed BF16 tests

// Packed BF16 maximum: a NaN half loses to a number (both NaN: NaN).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// 0xFFFF in each half where a >= b as BF16 numbers, else 0 (a NaN half: 0).
__device__ __forceinline__ uint32_t bge2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// The BF16 bits of the value whose order key is `key` (0x7F..0xFF80).
__device__ __forceinline__ uint32_t key_value(uint32_t key) {
    return key >= 0x8000u ? key - 0x8000u : key ^ 0xFFFFu;
}

// The order key of 16-bit BF16 bits x: x ^ (x < 0 ? 0xFFFF : 0x8000).
__device__ __forceinline__ uint32_t value_key(uint32_t x) {
    return x ^ ((x & 0x8000u) ? 0xFFFFu : 0x8000u);
}

// The packed compare operand of cut c: a non-NaN value x has key(x) >= c
// exactly when x >= value(c) as a BF16 number, for every c in [key(-inf),
// key(+inf)] except key(+0), where the numbers -0 and +0 compare equal. So c is
// clamped into that range (no eligible key lies outside it) and key(+0) is
// lowered to key(-0): a lower cut is still a cut (more keys at or above it).
__device__ __forceinline__ uint32_t cut_operand(uint32_t &c) {
    c = min(max(c, KEY_NEG_INF), KEY_POS_INF);
    if (c == 0x8000u) c = 0x7FFFu;
    const uint32_t v = key_value(c);
    return v | (v << 16);
}

// Bit i of the result: the low half of word i of r is >= the operand; bit 4 + i:
// its high half.
__device__ __forceinline__ uint32_t mask8(const uint4 &r, uint32_t cv) {
    const uint32_t t = (bge2(r.x, cv) & 0x00010001u) | (bge2(r.y, cv) & 0x00020002u) |
                       (bge2(r.z, cv) & 0x00040004u) | (bge2(r.w, cv) & 0x00080008u);
    return (t | (t >> 12)) & 0xFFu;
}

// The key of the larger half of a packed pair (0 for NaN).
__device__ __forceinline__ uint32_t top_key(uint32_t m) {
    const uint32_t x = bmax2(m, __byte_perm(m, 0, 0x1032)) & 0xFFFFu;
    return (x & 0x7FFFu) > 0x7F80u ? 0u : value_key(x);
}

__device__ __forceinline__ uint32_t vec_bmax(const uint4 &r) {
    return bmax2(bmax2(r.x, r.y), bmax2(r.z, r.w));
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

}  // namespace topk
