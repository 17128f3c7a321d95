// topk_ragged.cu -- deterministic exact ragged top-k for GB300 (sm_103a).
//
// The selection is the one sglang PR #31115 "Add opt-in deterministic
// CuTe-DSL DSA top-k backend" defines (PR summary, Modifications, hardening
// commit): canonical order score descending / index ascending on
// bitwise-equal scores, the smallest-index subset of the boundary tie set,
// no dropped candidates, -1 padding, and the bitwise total order on fp32
// patterns.  The pages' own kernel (one 512-thread CTA per row, an 8-bit
// coarse histogram, radix refinement, an index radix pass for ties, a
// bitonic sort of 24-bit-index composites) was written for other hardware;
// this file keeps its semantics and restructures the work for GB300:
//
//   * each thread-block cluster of C CTAs (C = 2..16, chosen on the host)
//     takes a group of rows, and every row a contiguous group of the
//     cluster's CTAs; each CTA owns a contiguous, 16-byte-aligned slice of
//     the row and stages as much of it as fits in shared memory (TMA bulk
//     copies), so the row is read from HBM once; the rest of a very long
//     slice is re-read from L2;
//   * an MSB-first radix select on the monotone uint32 order key with digits
//     of 11, 11 and 10 bits; per-CTA histograms use shared-memory atomics
//     (colliding lanes are merged by the hardware), and after a cluster
//     barrier every CTA of the row's group pulls the group's histograms over
//     distributed shared memory and makes the same threshold search, so the
//     k-th key T, the count above it and the count needed from its tie set
//     are exact integers, independent of scheduling;
//   * every entry above T is a winner; entries equal to T are ranked by
//     index with ordered per-warp / per-CTA prefix counts (the tie set is
//     taken in index order, so its first r members are the smallest indices,
//     and they already sit in canonical order after the winners);
//   * the winners are gathered into the row's leader CTA as unique
//     (key << 32 | ~index) composites and sorted descending in shared memory
//     (a counting bucket sort, bitonic only on skewed keys); the row is
//     written with coalesced stores.
//
// Batches of many rows (or of short ones) take a one-CTA-per-row kernel
// instead (topk_row_kernel): rows of up to 4096 scores are ranked from
// registers by one bucket pass split at +0.0, longer ones by the same radix
// select over shared memory.
//
// The same file holds the operations around the selection: the page-table
// transform of the output (a pass over each finished row, in the same
// launch), the per-row tie / plateau statistics (topk_stats_kernel and its
// cluster form), and, from indexer_scores.cuh, the lightning-indexer scores
// on the tcgen05 tensor cores.
//
// Nothing is allocated; the only global state is a status word for data
// errors.  Cross-CTA synchronisation uses hardware cluster barriers, and
// every mbarrier wait has an iteration limit.  Every kernel starts with a
// programmatic-dependent-launch wait, so it touches no global memory before
// the grids ahead of it in the stream have finished.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "plan.h"
#include "topk_ragged.h"

namespace {

using topk_plan::CCtrl;
using topk_plan::Ctrl;
using topk_plan::kBins;   // 11-bit digits (the last level uses 10 bits)
using topk_plan::kShortQuads;
using topk_plan::kShortScores;
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr uint32_t kNegInfBits = 0xFF800000u;
constexpr int kMaxDevices = 64;

__device__ uint32_t g_status;          // OR of TOPK_DEV_* bits

struct Params {
    const float *scores;
    int64_t n_scores;
    const int32_t *row_starts;
    const int32_t *lengths;
    int32_t *out_idx;
    float *out_val;
    int32_t B, k, offset_mode;
    int32_t stage_cap;   // scores per CTA kept in shared memory (multiple of 4)
    int32_t win_cap;     // winner slots in the leader (power of two >= k - 1)
    int32_t off_win;     // byte offset of the winner array in dynamic smem
    int32_t off_keys;    // byte offset of the staged keys in dynamic smem
    const int32_t *page_table;   // null, or B rows of pt_stride page numbers
    int64_t pt_stride;
    int32_t page_size;
    int32_t page_shift;          // log2(page_size) when a power of two, else -1
    int32_t ahead;               // row kernel: L2 prefetch distance in rows (0: none)
};

// Per-CTA control blocks (Ctrl, CCtrl) sit at the start of dynamic shared
// memory; plan.h defines them beside the launch planner that sizes them.

// ------------------------------------------------------------------------- //
// Order key: fp32 bits -> uint32 whose unsigned order is the bitwise total
// order (negative patterns are inverted, non-negative ones get the top bit).
// ------------------------------------------------------------------------- //
__device__ __forceinline__ uint32_t order_key(uint32_t u)
{
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

__device__ __forceinline__ uint32_t key_bits(uint32_t key)
{
    return (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
}

constexpr uint32_t kNegInfKey = 0x007FFFFFu;   // order key of -inf

// Writes one selected entry at output place pos: its index (plus the row
// offset) and its score, or -1 / -inf when the exclusion flag leaves the
// score out.  Excluded scores (-inf and every negative NaN: keys at or
// below that of -inf) rank after all others, so they fill a tail of the
// selection and the row stays front-packed.
__device__ __forceinline__ void put_out(int32_t *oi, float *ov, uint32_t pos, int64_t idx_offset, int32_t j,
                                        uint32_t key, bool excl)
{
    const bool drop = excl && key <= kNegInfKey;
    oi[pos] = drop ? -1 : (int32_t)(idx_offset + j);
    if (ov) ov[pos] = __uint_as_float(drop ? kNegInfBits : key_bits(key));
}

// ------------------------------------------------------------------------- //
// Cluster / DSMEM primitives (inline PTX).
// ------------------------------------------------------------------------- //
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync()
{
    cluster_arrive();
    cluster_wait();
}

// Shared::cluster address of `p` (a local shared-memory pointer) in CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t rank)
{
    uint32_t local = (uint32_t)__cvta_generic_to_shared(p);
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    return remote;
}

__device__ __forceinline__ uint32_t dsmem_ld(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void dsmem_ld_bins(uint32_t addr, uint32_t (&v)[2])
{
    asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(addr) : "memory");
}

__device__ __forceinline__ void dsmem_ld_bins(uint32_t addr, uint32_t (&v)[4])
{
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(addr) : "memory");
}

// ------------------------------------------------------------------------- //
// mbarrier and bulk-copy (TMA) primitives (inline PTX).
// ------------------------------------------------------------------------- //
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// mbarrier.init of one barrier.  The thread that initialises a set of
// barriers calls mbar_init_fence() once after the last of them, before any
// copy or commit may complete on one.
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes the barriers initialised so far visible to the bulk-copy (async)
// proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Global -> shared bulk copy that completes `bytes` of transactions on
// `bar`.  dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Bounded wait for phase `parity` of `bar`.  A copy that never lands is a
// hardware or library fault: the status word records it, and a second
// bounded wait gives the copies in flight time to finish before the CTA
// goes on, so that no late copy can land in reused shared memory.
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ void mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit = kWaitLimit)
{
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return;
    atomicOr(&g_status, TOPK_DEV_INTERNAL);
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return;
}

// The bounded wait above, on an mbarrier that nothing ever completes: one
// thread polls it `limit` times twice, the status word gets
// TOPK_DEV_INTERNAL, and the CTA exits (nothing is in flight).
__global__ void wait_probe_kernel(uint32_t limit)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
        mbar_wait_bounded(&bar, 0, limit);
    }
}

// Programmatic dependent launch: the next grid in the stream may be staged
// once every CTA of this one has started, and no CTA touches global memory
// before the grids ahead of it in the stream have finished and their writes
// are visible.
__device__ __forceinline__ void grid_dependency_enter()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------------- //
// Warp / block helpers.
// ------------------------------------------------------------------------- //
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Inclusive scan over the CTA in thread order.  `sm` holds 32 words; the
// caller must not reuse it before the next __syncthreads.
template <int THREADS>
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t x, uint32_t *sm)
{
    constexpr int NW = THREADS / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x = warp_incl_scan(x);
    if (lane == 31) sm[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < NW ? sm[lane] : 0u;
        w = warp_incl_scan(w);
        if (lane < NW) sm[lane] = w;
    }
    __syncthreads();
    if (warp > 0) x += sm[warp - 1];
    return x;
}

// Inclusive scan over the CTA in thread order with one barrier: each warp
// adds up the totals of the warps before it with a warp reduction.  `sm`
// holds NW words and must not be reused before the next __syncthreads.
template <int THREADS>
__device__ __forceinline__ uint32_t block_incl_scan1(uint32_t x, uint32_t *sm, uint32_t &total)
{
    constexpr int NW = THREADS / 32;
    static_assert(NW <= 32, "one warp total per lane");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t incl = warp_incl_scan(x);
    if (lane == 31) sm[warp] = incl;
    __syncthreads();
    const uint32_t v = lane < NW ? sm[lane] : 0u;
    total = __reduce_add_sync(kFull, v);
    return __reduce_add_sync(kFull, lane < warp ? v : 0u) + incl;
}

// Histogram increment: one shared-memory atomic add of 1 per lane.  The build
// switch TOPK_MATCH_AGGREGATE=1 (off in the library, kept for the measured
// comparison) merges the lanes of a warp that hit one bin with
// __match_any_sync first and lets one of them add the group's count; on the
// decode and causal prefill batches that form was slower (the plain atomic
// is merged by the shared-memory unit, the match costs a warp-wide
// instruction per increment).
#ifndef TOPK_MATCH_AGGREGATE
#define TOPK_MATCH_AGGREGATE 0
#endif
__device__ __forceinline__ void hist_inc(uint32_t *hist, uint32_t bin)
{
#if TOPK_MATCH_AGGREGATE
    uint32_t lt;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
    const uint32_t peers = __match_any_sync(__activemask(), bin);
    if ((peers & lt) == 0u) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
#else
    atomicAdd(&hist[bin], 1u);
#endif
}

__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t digit, bool valid)
{
    if (valid) hist_inc(hist, digit);
}

// ------------------------------------------------------------------------- //
// A CTA's slice of its row, in "slots": slot 0 is 16-byte aligned in global
// memory; valid slots are [off0, end); quads (4 slots) in [bq0, bq1) lie
// entirely inside the row and are read with one 16-byte load; quads below sq
// are staged in shared memory.
// ------------------------------------------------------------------------- //
struct Slice {
    const float *gptr;   // scores + global index of slot 0
    int32_t off0, end;   // valid slot range
    int32_t bq0, bq1;    // full quads inside the row
    int32_t nq;          // quads covering [0, end)
    int32_t sq;          // staged quads
    int32_t jbase;       // row-local index of slot 0 (may be -3..0)
};

__device__ __forceinline__ uint32_t quad_mask(const Slice &s, int q)
{
    int lo = s.off0 - 4 * q, hi = s.end - 4 * q;
    lo = lo < 0 ? 0 : lo;
    hi = hi > 4 ? 4 : hi;
    return hi > lo ? (((1u << hi) - 1u) & ~((1u << lo) - 1u)) : 0u;
}

__device__ __forceinline__ uint4 load_quad_global(const Slice &s, int q, uint32_t &m)
{
    if (q >= s.bq0 && q < s.bq1) {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(s.gptr) + q);
        m = 0xFu;
        return make_uint4(order_key(__float_as_uint(f.x)), order_key(__float_as_uint(f.y)),
                          order_key(__float_as_uint(f.z)), order_key(__float_as_uint(f.w)));
    }
    m = quad_mask(s, q);
    uint32_t e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        e[i] = ((m >> i) & 1u) ? order_key(__float_as_uint(__ldg(s.gptr + 4 * q + i))) : 0u;
    return make_uint4(e[0], e[1], e[2], e[3]);
}

__device__ __forceinline__ uint4 load_quad(const Slice &s, const uint32_t *keys, int q, uint32_t &m)
{
    if (q < s.sq) {
        m = quad_mask(s, q);
        return reinterpret_cast<const uint4 *>(keys)[q];
    }
    return load_quad_global(s, q, m);
}

// ------------------------------------------------------------------------- //
// Threshold search: given a histogram h over kBins digits (larger digit =
// larger key) and r >= 1 entries still to take, find the bin b with
// sum(h[> b]) < r <= sum(h[>= b]).  The single owning thread returns true
// with (b, sum(h[> b]), h[b]); the caller publishes and synchronises.
// Each thread owns BPT consecutive bins, read as 16-byte vectors.
// ------------------------------------------------------------------------- //
template <int THREADS>
__device__ __forceinline__ void load_bins(const uint32_t *h, int lo, uint32_t (&v)[kBins / THREADS])
{
    constexpr int BPT = kBins / THREADS;
    if constexpr (BPT % 4 == 0) {
#pragma unroll
        for (int i = 0; i < BPT; i += 4) {
            const uint4 x = *reinterpret_cast<const uint4 *>(h + lo + i);
            v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < BPT; i += 2) {
            const uint2 x = *reinterpret_cast<const uint2 *>(h + lo + i);
            v[i] = x.x; v[i + 1] = x.y;
        }
    }
}

template <int THREADS>
__device__ __forceinline__ bool find_bin(const uint32_t *h, uint32_t r, uint32_t *sm,
                                         uint32_t &digit, uint32_t &gt, uint32_t &cnt)
{
    constexpr int BPT = kBins / THREADS;
    const int lo = kBins - ((int)threadIdx.x + 1) * BPT;   // thread 0 owns the top bins
    uint32_t v[BPT];
    load_bins<THREADS>(h, lo, v);
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) sum += v[i];
    const uint32_t incl = block_incl_scan<THREADS>(sum, sm);
    const uint32_t excl = incl - sum;
    bool mine = false;
    if (excl < r && r <= incl) {
        uint32_t acc = excl;
#pragma unroll
        for (int i = BPT - 1; i >= 0; --i) {   // descending bins
            if (!mine && acc + v[i] >= r) {
                mine = true;
                digit = (uint32_t)(lo + i);
                gt = acc;
                cnt = v[i];
            }
            acc += v[i];
        }
    }
    return mine;
}

// find_bin over NB bins (NB / THREADS a multiple of 2 per thread).
template <int THREADS, int NB>
__device__ __forceinline__ bool find_bin_nb(const uint32_t *h, uint32_t r, uint32_t *sm, uint32_t &digit,
                                            uint32_t &gt)
{
    constexpr int BPT = NB / THREADS;
    static_assert(BPT % 2 == 0, "two or more bins per thread");
    const int lo = NB - ((int)threadIdx.x + 1) * BPT;   // thread 0 owns the top bins
    uint32_t v[BPT];
#pragma unroll
    for (int i = 0; i < BPT; i += 2) {
        const uint2 x = *reinterpret_cast<const uint2 *>(h + lo + i);
        v[i] = x.x;
        v[i + 1] = x.y;
    }
    uint32_t sum = 0, total;
#pragma unroll
    for (int i = 0; i < BPT; ++i) sum += v[i];
    const uint32_t incl = block_incl_scan1<THREADS>(sum, sm, total);
    bool mine = false;
    if (incl - sum < r && r <= incl) {
        uint32_t acc = incl - sum;
#pragma unroll
        for (int i = BPT - 1; i >= 0; --i) {
            if (!mine && acc + v[i] >= r) {
                mine = true;
                digit = (uint32_t)(lo + i);
                gt = acc;
            }
            acc += v[i];
        }
    }
    return mine;
}

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ------------------------------------------------------------------------- //
// Descending bitonic sort of n = power of two composites (the fallback of
// bucket_sort_desc for pathologically skewed key distributions).
// ------------------------------------------------------------------------- //
template <int THREADS>
__device__ void bitonic_desc(uint64_t *a, uint32_t n)
{
    for (uint32_t size = 2; size <= n; size <<= 1) {
        for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (uint32_t i = threadIdx.x; i < (n >> 1); i += THREADS) {
                const uint32_t lo = 2 * i - (i & (stride - 1));
                const uint32_t hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const uint64_t x = a[lo], y = a[hi];
                if ((x < y) == desc) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

// ------------------------------------------------------------------------- //
// 64-bit inclusive block scan (two 32-bit counters packed in one word); the
// CTA-wide total is returned in `total`.  `sm` holds 32 64-bit words.
// ------------------------------------------------------------------------- //
template <int THREADS>
__device__ __forceinline__ uint64_t block_incl_scan64(uint64_t x, uint64_t *sm, uint64_t &total)
{
    constexpr int NW = THREADS / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint64_t w = lane < NW ? sm[lane] : 0ull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NW) sm[lane] = w;
    }
    __syncthreads();
    if (warp > 0) x += sm[warp - 1];
    total = sm[NW - 1];
    return x;
}

// ------------------------------------------------------------------------- //
// Sort the n unique composites (key << 32 | ~index) of a[0..n), all with
// keys in [kmin, kmax], into canonical order (composite descending) and
// write them to the output row.  The key range is cut into kBins buckets of
// 2^s keys; bucket sizes come from a shared-memory histogram and are laid
// out from the top bucket down by a scan; every composite is dropped into its
// bucket (order inside a bucket is arbitrary) and its final position is the
// bucket start plus the number of bucket members above it, so the result
// depends only on the composites.  Work is n + sum(m_b^2); when the buckets
// are too skewed for that to stay small the function sorts with a bitonic
// network instead.  Only the first n_out places are written.  b[] is
// scratch for n composites, cur[] kBins words.
// ------------------------------------------------------------------------- //
template <int THREADS>
__device__ void sort_and_write(uint64_t *a, uint64_t *b, int n, int n_out, int cap_pow2, uint32_t kmin,
                               uint32_t kmax, uint32_t *cur, uint64_t *sm64, int32_t *oi, float *ov,
                               int64_t idx_offset, bool excl)
{
    constexpr int BPT = kBins / THREADS;
    const int tid = threadIdx.x;
    const uint32_t range = kmax - kmin;
    const int s = max(0, (32 - __clz(range)) - 11);
    for (int i = tid; i < kBins; i += THREADS) cur[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += THREADS) hist_inc(cur, ((uint32_t)(a[i] >> 32) - kmin) >> s);
    __syncthreads();
    const int lo = kBins - (tid + 1) * BPT;
    uint32_t v[BPT];
    load_bins<THREADS>(cur, lo, v);
    uint64_t pair = 0;   // (sum of squares << 32) | count
#pragma unroll
    for (int i = 0; i < BPT; ++i) pair += ((uint64_t)(v[i] * v[i]) << 32) | v[i];
    uint64_t total;
    const uint64_t incl = block_incl_scan64<THREADS>(pair, sm64, total);
    uint32_t run = (uint32_t)(incl - pair);
    const uint32_t total_sq = (uint32_t)(total >> 32);
    if (total_sq > 256u * (uint32_t)n + 4096u) {
        int n2 = 1;
        while (n2 < n) n2 <<= 1;
        if (n2 > cap_pow2) n2 = cap_pow2;   // n <= cap_pow2 always
        for (int i = n + tid; i < n2; i += THREADS) a[i] = 0ull;
        __syncthreads();
        bitonic_desc<THREADS>(a, (uint32_t)n2);
        for (int p = tid; p < n_out; p += THREADS) {
            const uint64_t c = a[p];
            put_out(oi, ov, (uint32_t)p, idx_offset, (int32_t)(~(uint32_t)c), (uint32_t)(c >> 32), excl);
        }
        return;
    }
#pragma unroll
    for (int i = BPT - 1; i >= 0; --i) {   // bucket starts, top bucket first
        cur[lo + i] = run;
        run += v[i];
    }
    __syncthreads();
    for (int i = tid; i < n; i += THREADS) {
        const uint64_t x = a[i];
        const uint32_t pos = atomicAdd(&cur[((uint32_t)(x >> 32) - kmin) >> s], 1u);
        b[pos] = x;
    }
    __syncthreads();
    // cur[d] is now the end of bucket d, and the start of bucket d is the
    // end of bucket d + 1 (buckets are laid out from the top digit down).
    for (int p = tid; p < n; p += THREADS) {
        const uint64_t x = b[p];
        const uint32_t d = ((uint32_t)(x >> 32) - kmin) >> s;
        const uint32_t st = d + 1 < (uint32_t)kBins ? cur[d + 1] : 0u;
        const uint32_t en = cur[d];
        uint32_t rank = 0;
        for (uint32_t q = st; q < en; ++q) rank += b[q] > x;
        const uint32_t pos = st + rank;
        if (pos < (uint32_t)n_out)
            put_out(oi, ov, pos, idx_offset, (int32_t)(~(uint32_t)x), (uint32_t)(x >> 32), excl);
    }
}

// ------------------------------------------------------------------------- //
// Short rows: one CTA per row with the whole row in registers (at most
// kShortQuads quads per thread).  Canonical order cuts a row at the order
// key of +0.0 into P (keys above it), the +0.0 entries and N (keys below
// it), and lists P in key order, then the +0.0 entries by index, then N in
// key order.  The non-zero entries are ranked together by one bucket pass
// over their own key range [kmin, kmax]: 2^nb buckets of 2^sh keys, about
// four per non-zero entry, bucket starts from a scan, every entry dropped
// into its bucket, and its place the bucket start plus the number of
// members of its bucket above it (composites are unique, so this is exact).
// When the row holds both signs, the bucket grid is shifted so that a bucket
// edge falls on +0.0's key: the start of the first bucket below it is then
// |P|.  Buckets that start at or after k are never output and are not
// ranked.  An N entry moves down by the +0.0 count; a +0.0 entry's place is
// |P| plus its ordinal in index order, from per-warp ballots.  When an
// output bucket is too big for member counting to stay cheap (heavy ties off
// +0.0) the function returns false with shared memory released and the
// general path runs.
//
// The counters are one 32-bit word per bucket (at most 4096 buckets), each
// histogram atomic a constant +1.
// ------------------------------------------------------------------------- //
constexpr int kShortMinWordsLog = 10;        // at least 1024 counter words
constexpr int kShortMaxWordsLog = 12;        // at most 4096 counter words (16 KB)
constexpr int kShortExtraBits = 2;           // about four buckets per non-zero entry
constexpr uint32_t kShortMaxBucket = 48;     // largest output bucket ranked by counting
// Build switch kept for the measured comparison of counter forms (off in
// the library): TOPK_SHORT_PACKED=1 packs two 16-bit counters into a word
// (twice the buckets, a variable increment of 1 or 1 << 16).  On the causal
// prefill batch (16384 rows, k = 2048) it ran slower than one-word counters
// with a constant increment.
#ifndef TOPK_SHORT_PACKED
#define TOPK_SHORT_PACKED 0
#endif
constexpr bool kShortPacked = TOPK_SHORT_PACKED;

// One quad of a short row as order keys, every slot outside the row read as
// the key of +0.0 (its bit in m is clear).
__device__ __forceinline__ uint4 load_quad_short(const Slice &s, int q, uint32_t &m)
{
    constexpr uint32_t kZ = 0x80000000u;
    if (q >= s.bq0 && q < s.bq1) {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(s.gptr) + q);
        m = 0xFu;
        return make_uint4(order_key(__float_as_uint(f.x)), order_key(__float_as_uint(f.y)),
                          order_key(__float_as_uint(f.z)), order_key(__float_as_uint(f.w)));
    }
    m = q < s.nq ? quad_mask(s, q) : 0u;
    uint32_t e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        e[i] = ((m >> i) & 1u) ? order_key(__float_as_uint(__ldg(s.gptr + 4 * q + i))) : kZ;
    return make_uint4(e[0], e[1], e[2], e[3]);
}

// Entries k_eff .. k of an output row as -1 (and -inf), 16-byte stores over
// the aligned middle.
__device__ __forceinline__ void pad_out(int32_t *oi, float *ov, int from, int to)
{
    if (from >= to) return;
    const int t = (int)threadIdx.x, nt = (int)blockDim.x;
    int a = from + (int)((4u - (uint32_t)(((uintptr_t)(oi + from) >> 2) & 3u)) & 3u);
    if (a > to) a = to;
    const int nv = (to - a) >> 2, tail = a + 4 * nv;
    if (t < a - from) oi[from + t] = -1;
    if (t < to - tail) oi[tail + t] = -1;
    int4 *o4 = reinterpret_cast<int4 *>(oi + a);
    for (int q = t; q < nv; q += nt) o4[q] = make_int4(-1, -1, -1, -1);
    if (ov)
        for (int p = from + t; p < to; p += nt) ov[p] = __uint_as_float(kNegInfBits);
}

// Exclusive scan over the CTA in thread order with one barrier: every warp
// adds up the totals of the warps before it.  `sm` holds NW words and must
// not be reused before the next __syncthreads.
template <int THREADS>
__device__ __forceinline__ uint32_t block_excl_scan1(uint32_t x, uint32_t *sm, uint32_t &total)
{
    constexpr int NW = THREADS / 32;
    static_assert(NW % 4 == 0, "warp totals read as 16-byte vectors");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t incl = warp_incl_scan(x);
    if (lane == 31) sm[warp] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < NW; w += 4) {
        const uint4 v = *reinterpret_cast<const uint4 *>(sm + w);
        before += (w < warp ? v.x : 0u) + (w + 1 < warp ? v.y : 0u) + (w + 2 < warp ? v.z : 0u) +
                  (w + 3 < warp ? v.w : 0u);
        all += v.x + v.y + v.z + v.w;
    }
    total = all;
    return before + incl - x;
}

template <int THREADS>
__device__ bool short_row(Ctrl &ctrl, unsigned char *area, uint32_t area_bytes, const Slice &s, uint32_t k_eff,
                          int64_t idx_offset, int32_t *oi, float *ov, int k, bool excl)
{
    constexpr int NW = THREADS / 32;
    constexpr uint32_t kZ = 0x80000000u;   // order key of +0.0
    constexpr bool PK = kShortPacked;
    constexpr int kMaxWords = 1 << kShortMaxWordsLog;
    constexpr int kBucketsPerWord = PK ? 2 : 1;
    static_assert(kShortQuads * NW <= 32, "one (quad round, warp) count per lane of warp 0");
    static_assert((1 << kShortMinWordsLog) % (4 * THREADS) == 0, "whole 16-byte word groups per thread");
    static_assert(kMaxWords / (4 * THREADS) <= 4, "at most four word groups per thread");
    uint32_t *cur = reinterpret_cast<uint32_t *>(area);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t lt = lanemask_lt();

    // Thread t holds quads t, t + THREADS, ...: index order is round u, then
    // warp, then lane, then slot.  Round u of a warp holds data iff
    // active(u); the test is warp-uniform.
    auto active = [&](int u) { return warp * 32 + u * THREADS < s.nq; };
    for (int i = tid; i < kMaxWords / 4; i += THREADS) reinterpret_cast<uint4 *>(cur)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) ctrl.sq = 0u;
    // Keys, the 16-bit masks of valid slots (vm) and of +0.0-keyed slots
    // (zm: the +0.0 entries and every slot outside the row), the range of
    // the non-zero keys, and the +0.0 count of each round (8 bits a round).
    uint32_t key[kShortQuads][4];
    uint32_t zm = 0, vm = 0, kmin = kFull, kmax = 0, zc = 0;
#pragma unroll
    for (int u = 0; u < kShortQuads; ++u) {
        key[u][0] = key[u][1] = key[u][2] = key[u][3] = kZ;
        if (!active(u)) continue;
        uint32_t m;
        const uint4 kk = load_quad_short(s, tid + u * THREADS, m);
        key[u][0] = kk.x; key[u][1] = kk.y; key[u][2] = kk.z; key[u][3] = kk.w;
        uint32_t z4 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t e = key[u][i];
            const bool z = e == kZ;
            z4 |= (uint32_t)z << i;
            kmin = min(kmin, z ? kFull : e);
            kmax = max(kmax, z ? 0u : e);
        }
        zm |= z4 << (4 * u);
        vm |= m << (4 * u);
        zc |= (uint32_t)__popc(z4 & m) << (8 * u);
    }
    const uint32_t nzm = vm & ~zm;   // non-zero entries
    kmin = __reduce_min_sync(kFull, kmin);
    kmax = __reduce_max_sync(kFull, kmax);
    const uint32_t nnz_w = __reduce_add_sync(kFull, (uint32_t)__popc(nzm));
    zc = __reduce_add_sync(kFull, zc);   // at most 128 a round: no carry between rounds
    if (lane == 0) {
        ctrl.part_min[warp] = kmin;
        ctrl.part_max[warp] = kmax;
        ctrl.part_p[warp] = nnz_w;
    }
    if (lane < kShortQuads) ctrl.warp_zeros[lane * NW + warp] = (zc >> (8 * lane)) & 0xFFu;
    __syncthreads();

    uint32_t nzmin = kFull, nzmax = 0, nnz = 0;
#pragma unroll
    for (int w = 0; w < NW; w += 4) {
        const uint4 a = *reinterpret_cast<const uint4 *>(&ctrl.part_min[w]);
        const uint4 b = *reinterpret_cast<const uint4 *>(&ctrl.part_max[w]);
        const uint4 c = *reinterpret_cast<const uint4 *>(&ctrl.part_p[w]);
        nzmin = min(min(nzmin, min(a.x, a.y)), min(a.z, a.w));
        nzmax = max(max(nzmax, max(b.x, b.y)), max(b.z, b.w));
        nnz += c.x + c.y + c.z + c.w;
    }
    if (tid == 0) ctrl.npart = nnz;   // lowered below to the first bucket start at or past k_eff
    // Bucket grid: 2^nb buckets (nb from the non-zero count, within the
    // area left beside the composites that are ranked), bucket d holding keys
    // base + [d << sh, (d + 1) << sh).
    const uint32_t need = min(nnz, k_eff + kShortMaxBucket);
    constexpr int kPk = PK ? 1 : 0;
    int nb = (32 - __clz(max(nnz, 2u) - 1u)) + kShortExtraBits;
    nb = min(max(nb, kShortMinWordsLog + kPk), kShortMaxWordsLog + kPk);
    while (nb > kShortMinWordsLog + kPk && (4u << (nb - kPk)) + 8u * need > area_bytes) --nb;
    const uint32_t nwords = 1u << (nb - kPk);
    uint64_t *buf = reinterpret_cast<uint64_t *>(area + 4u * nwords);
    const uint32_t buf_cap = (area_bytes - 4u * nwords) / 8u;
    int sh = max(0, (32 - __clz(nzmax - nzmin)) - nb);
    uint32_t base = nzmin, c0 = 0;   // c0: first bucket above +0.0 when the row has both signs
    const bool split = nnz && nzmin < kZ && nzmax > kZ;
    if (split) {
        c0 = (kZ - nzmin + (1u << sh) - 1u) >> sh;
        base = kZ - (c0 << sh);
        if ((nzmax - base) >> sh >> nb) {
            ++sh;
            c0 = (kZ - nzmin + (1u << sh) - 1u) >> sh;
            base = kZ - (c0 << sh);
        }
    }
    // Counter word and increment of bucket d.
    auto word_of = [&](uint32_t d) { return PK ? d >> 1 : d; };
    auto inc_of = [&](uint32_t d) { return PK ? 1u << ((d & 1u) << 4) : 1u; };
    if (nnz) {
#pragma unroll
        for (int u = 0; u < kShortQuads; ++u) {
            if (!active(u)) continue;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if ((nzm >> (4 * u + i)) & 1u) {
                    const uint32_t d = (key[u][i] - base) >> sh;
                    if (PK)
                        atomicAdd(&cur[word_of(d)], inc_of(d));
                    else
                        hist_inc(cur, d);
                }
            }
        }
    }
    __syncthreads();
    uint32_t P = 0;
    if (nnz) {
        // Bucket starts, top bucket first (in a packed word the high half
        // is the higher bucket).  Thread t scans nch groups of four words,
        // thread 0 the top ones; the sums of a word's two halves never carry.
        const int nch = (int)nwords / (4 * THREADS);
        const int w0 = (int)nwords - (tid + 1) * 4 * nch;
        uint4 v[4];
        uint32_t sum = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (c < nch) {
                v[c] = *reinterpret_cast<const uint4 *>(cur + w0 + 4 * c);
                sum += v[c].x + v[c].y + v[c].z + v[c].w;
            }
        }
        const uint32_t tot = PK ? (sum >> 16) + (sum & 0xFFFFu) : sum;
        uint32_t all;
        const uint32_t run_in = block_excl_scan1<THREADS>(tot, ctrl.scan, all);
        // np: the first bucket start at or past k_eff in this thread's
        // words; mx: the largest bucket.
        uint32_t run = run_in, mx = 0, np = kFull;
        auto start_of = [&](uint32_t x) {   // word of counts -> word of starts
            if (PK) {
                const uint32_t hi = x >> 16, st = run * 0x10001u + hi;
                const uint32_t lo_st = run + hi;
                np = min(np, run >= k_eff ? run : kFull);
                np = min(np, lo_st >= k_eff ? lo_st : kFull);
                run = lo_st + (x & 0xFFFFu);
                mx = __vmaxu2(mx, x);
                return st;
            }
            const uint32_t st = run;
            np = min(np, st >= k_eff ? st : kFull);
            run += x;
            mx = max(mx, x);
            return st;
        };
#pragma unroll
        for (int c = 3; c >= 0; --c) {
            if (c < nch) {
                v[c].w = start_of(v[c].w);
                v[c].z = start_of(v[c].z);
                v[c].y = start_of(v[c].y);
                v[c].x = start_of(v[c].x);
                *reinterpret_cast<uint4 *>(cur + w0 + 4 * c) = v[c];
            }
        }
        // Entries in the buckets that start below k_eff (the ones ranked):
        // the start of the first bucket at or past k_eff, or every
        // non-zero entry.
        np = __reduce_min_sync(kFull, np);
        if (lane == 0 && np < nnz) atomicMin(&ctrl.npart, np);
        // The largest bucket among those ranked (the words of the thread
        // that crosses k_eff may add a few that are not: a bound only).
        uint32_t mb = run_in < k_eff ? (PK ? max(mx >> 16, mx & 0xFFFFu) : mx) : 0u;
        mb = __reduce_max_sync(kFull, mb);
        if (lane == 0 && mb) atomicMax(&ctrl.sq, mb);
        __syncthreads();
        if (split) {
            const uint32_t d = c0 - 1, w = cur[word_of(d)];
            P = PK ? (((d & 1u) ? (w >> 16) : w) & 0xFFFFu) : w;
        } else {
            P = nzmin > kZ ? nnz : 0u;
        }
    } else {
        __syncthreads();
    }
    const uint32_t npart = ctrl.npart;
    if (npart > buf_cap || ctrl.sq > kShortMaxBucket) {   // CTA-uniform
        __syncthreads();
        return false;
    }
    // Exclusive bases of the (round, warp) +0.0 counts in index order, and
    // the row's +0.0 total, scanned by every warp for itself.
    const uint32_t zt = ctrl.warp_zeros[lane];
    const uint32_t zti = warp_incl_scan(zt);
    const uint32_t Zc = __shfl_sync(kFull, zti, 31), zex = zti - zt;
    // Indices are written as 32-bit sums (the output is int32).
    const int32_t off32 = (int32_t)idx_offset;
    const bool plain = !excl && ov == nullptr;   // CTA-uniform
    if (npart) {
#pragma unroll
        for (int u = 0; u < kShortQuads; ++u) {
            if (!active(u)) continue;
            const uint32_t nj0 = ~(uint32_t)(s.jbase + 4 * (tid + u * THREADS));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if ((nzm >> (4 * u + i)) & 1u) {
                    const uint32_t e = key[u][i];
                    const uint32_t d = (e - base) >> sh;
                    uint32_t pos;
                    if (PK) {
                        const uint32_t hs = (d & 1u) << 4;
                        pos = (atomicAdd(&cur[d >> 1], 1u << hs) >> hs) & 0xFFFFu;
                    } else {
                        pos = atomicAdd(&cur[d], 1u);
                    }
                    if (pos < npart) buf[pos] = ((uint64_t)e << 32) | (uint64_t)(nj0 - (uint32_t)i);
                }
            }
        }
    }
    // The +0.0 entries go to P + their ordinal in index order.
    if (Zc > 0 && P < k_eff) {
#pragma unroll
        for (int u = 0; u < kShortQuads; ++u) {
            if (!active(u)) continue;
            const uint32_t z = (zm & vm) >> (4 * u) & 0xFu;
            uint32_t ord = P + __shfl_sync(kFull, zex, u * NW + warp);
            if (ord >= k_eff || !__any_sync(kFull, z)) continue;
#pragma unroll
            for (int i = 0; i < 4; ++i) ord += (uint32_t)__popc(__ballot_sync(kFull, (z >> i) & 1u) & lt);
            const int32_t j0 = off32 + s.jbase + 4 * (tid + u * THREADS);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if ((z >> i) & 1u) {
                    if (ord < k_eff) {
                        oi[ord] = j0 + i;
                        if (ov) ov[ord] = 0.0f;
                    }
                    ++ord;
                }
            }
        }
    }
    if (npart) {
        __syncthreads();
        // Bucket d's counter now holds its end, and the start of bucket d
        // is the end of bucket d + 1.
        const uint32_t top = kBucketsPerWord * nwords;
#pragma unroll 1
        for (uint32_t x = tid; x < npart; x += THREADS) {
            const uint64_t c = buf[x];
            const uint32_t e = (uint32_t)(c >> 32);
            const uint32_t d = (e - base) >> sh;
            uint32_t st, en;
            if (PK) {
                const uint32_t w = cur[d >> 1];
                en = (d & 1u) ? (w >> 16) : (w & 0xFFFFu);
                st = (d & 1u) ? (d + 1 < top ? cur[(d + 1) >> 1] & 0xFFFFu : 0u) : (w >> 16);
            } else {
                en = cur[d];
                st = d + 1 < top ? cur[d + 1] : 0u;
            }
            uint32_t pos = st, y = st;
#pragma unroll 1
            for (; y + 1 < en; y += 2) pos += (uint32_t)(buf[y] > c) + (uint32_t)(buf[y + 1] > c);
            if (y < en) pos += buf[y] > c;
            if (e < kZ) pos += Zc;
            if (pos < k_eff) {
                if (plain)
                    oi[pos] = off32 + (int32_t)(~(uint32_t)c);
                else
                    put_out(oi, ov, pos, idx_offset, (int32_t)(~(uint32_t)c), e, excl);
            }
        }
    }
    pad_out(oi, ov, (int)k_eff, k);
    return true;
}

// The page-table transform of a finished output row, in place: every
// in-row index j becomes pages[j / page_size] * page_size + j % page_size
// (-1 stays -1).  The caller makes the row's writes visible first.
// One in-row index through the page table (-1 stays -1).  Slots fit int32
// by contract, so 32-bit arithmetic is exact.
template <bool POW2>
__device__ __forceinline__ int32_t page_slot(int32_t j, const int32_t *pages, int32_t page_size, int32_t page_shift)
{
    if (j < 0) return j;
    if (POW2)
        return (int32_t)(((uint32_t)__ldg(pages + (j >> page_shift)) << page_shift) | (uint32_t)(j & (page_size - 1)));
    const int32_t pg = j / page_size;
    return __ldg(pages + pg) * page_size + (j - pg * page_size);
}

// The row's first n entries through the page table, four per 16-byte access
// when the row is 16-byte aligned (the entries from n up to the next
// multiple of four are -1 padding when k is a multiple of four), two
// accesses in flight per thread.
template <bool POW2>
__device__ __forceinline__ void page_map_entries(int32_t *oi, int n, int k, const int32_t *pages, int32_t page_size,
                                                 int32_t page_shift)
{
    const int nt = (int)blockDim.x;
    if ((k & 3) == 0 && ((uintptr_t)oi & 15u) == 0) {
        int4 *o4 = reinterpret_cast<int4 *>(oi);
        const int nq = (n + 3) >> 2;
        for (int q0 = (int)threadIdx.x; q0 < nq; q0 += 2 * nt) {
            int4 v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) v[u] = q0 + u * nt < nq ? o4[q0 + u * nt] : make_int4(-1, -1, -1, -1);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                v[u].x = page_slot<POW2>(v[u].x, pages, page_size, page_shift);
                v[u].y = page_slot<POW2>(v[u].y, pages, page_size, page_shift);
                v[u].z = page_slot<POW2>(v[u].z, pages, page_size, page_shift);
                v[u].w = page_slot<POW2>(v[u].w, pages, page_size, page_shift);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (q0 + u * nt < nq) o4[q0 + u * nt] = v[u];
        }
        return;
    }
    for (int q = (int)threadIdx.x; q < n; q += nt) oi[q] = page_slot<POW2>(oi[q], pages, page_size, page_shift);
}

// The page-table transform of a finished output row, in place: every
// in-row index j becomes pages[j / page_size] * page_size + j % page_size.
// The caller makes the row's writes visible to the CTA first.
__device__ __forceinline__ void page_map_row(const Params &p, int row, int32_t *oi, int n)
{
    const int32_t *pages = p.page_table + (int64_t)row * p.pt_stride;
    if (p.page_shift >= 0)
        page_map_entries<true>(oi, n, p.k, pages, p.page_size, p.page_shift);
    else
        page_map_entries<false>(oi, n, p.k, pages, p.page_size, p.page_shift);
}

// Quads of warp `warp`'s contiguous segment of the slice.
struct WarpSeg {
    int q0, q1;
};

template <int THREADS>
__device__ __forceinline__ WarpSeg warp_segment(int nq, int warp)
{
    constexpr int NW = THREADS / 32;
    const int per = (nq + NW - 1) / NW;
    const int q0 = min(nq, warp * per);
    return {q0, min(nq, q0 + per)};
}

// Row assignment of a grouped cluster: every CTA of the cluster computes it
// from the row lengths alone, so all of them agree.  Rows are ranked by
// valid length (descending, index ascending); rank t goes to cluster
// snake(t) (0..G-1, then G-1..0, ...), which spreads long rows over the
// clusters; inside a cluster the CTAs are dealt to its rows in proportion to
// their lengths (at least one each), so every CTA gets a similar slice.
struct RowGroup {
    int row;        // my row, or -1 when the cluster has no row with work
    uint32_t g0;    // cluster rank of the group's first CTA (its leader)
    uint32_t gsize; // CTAs working on the row
    int32_t start;  // the row's row_starts and valid length
    int32_t len;
};

__device__ __forceinline__ bool row_window_ok(const Params &p, int i, int64_t &len)
{
    const int64_t rs = p.row_starts[i];
    len = p.lengths[i];
    if (len < 0) len = 0;
    if (len >= (int64_t)TOPK_RAGGED_MAX_LEN) return false;
    return rs >= 0 && rs + len <= p.n_scores;
}

template <int THREADS>
__device__ RowGroup assign_rows(const Params &p, uint32_t crank, uint32_t csize, uint32_t *scratch,
                                uint32_t *slot)
{
    const int tid = threadIdx.x;
    const int B = p.B;   // at most 512 (the planner's cluster shapes hold fewer CTAs)
    const int G = (int)(gridDim.x / csize), cid = (int)(blockIdx.x / csize);
    uint32_t *eff = scratch;              // B valid lengths (0: nothing to select)
    uint32_t *starts = scratch + 512;     // B row starts
    uint32_t *by_rank = scratch + 1024;   // row index of every rank
    if (B <= 64) {
        // Up to 64 rows: warp 0 alone loads them (rows lane and lane + 32)
        // and ranks them with a bitonic sort of (length << 6 | 63 - row),
        // descending: length descending, row ascending.
        if (tid < 32) {
            const int lane = tid;
            uint32_t a[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                a[h] = 0u;
                if (i < B) {
                    int64_t len;
                    const uint32_t e = row_window_ok(p, i, len) ? (uint32_t)len : 0u;
                    eff[i] = e;
                    starts[i] = (uint32_t)p.row_starts[i];
                    a[h] = (e << 6) | (uint32_t)(63 - i);
                }
            }
#pragma unroll
            for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
                for (int j = k >> 1; j > 0; j >>= 1) {
                    if (j == 32) {   // elements lane and lane + 32, in one lane
                        const uint32_t hi = max(a[0], a[1]), lo = min(a[0], a[1]);
                        a[0] = hi;
                        a[1] = lo;
                    } else {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int i = lane + 32 * h;
                            const uint32_t o = __shfl_xor_sync(kFull, a[h], j);
                            // Blocks with (i & k) == 0 run descending.
                            const bool keep_max = ((i & j) == 0) == ((i & k) == 0);
                            a[h] = keep_max ? max(a[h], o) : min(a[h], o);
                        }
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (lane + 32 * h < B) by_rank[lane + 32 * h] = 63u - (a[h] & 63u);
            __syncwarp();
        }
    } else {
        for (int i = tid; i < B; i += THREADS) {
            int64_t len;
            eff[i] = row_window_ok(p, i, len) ? (uint32_t)len : 0u;
            starts[i] = (uint32_t)p.row_starts[i];
        }
        for (int i = B + tid; i < ((B + 3) & ~3); i += THREADS) eff[i] = 0u;   // pad to whole vectors
        __syncthreads();
        for (int i = tid; i < B; i += THREADS) {
            const uint32_t e = eff[i];
            int rank = 0;
            for (int j = 0; j < B; j += 4) {
                const uint4 q = *reinterpret_cast<const uint4 *>(eff + j);
                rank += (q.x > e || (q.x == e && j < i)) + (q.y > e || (q.y == e && j + 1 < i)) +
                        (q.z > e || (q.z == e && j + 2 < i)) + (q.w > e || (q.w == e && j + 3 < i));
            }
            by_rank[rank] = (uint32_t)i;
        }
        __syncthreads();
    }
    if (tid < 32) {
        // The cluster's rows, one per lane of warp 0, in the order they are
        // dealt: lane i holds rank t_i (the pair of block i / 2), and t_i
        // grows with i, so the cluster's rows are lanes 0 .. m-1, and (ranks
        // being sorted by length) the rows with work come first.  A cluster
        // holds at most csize of them (the planner guarantees it).
        const int lane = tid;
        const int t0 = (lane >> 1) * 2 * G;
        const int t = (lane & 1) ? t0 + 2 * G - 1 - cid : t0 + cid;
        const bool exists = lane < 16 && t < B;
        const uint32_t row_i = exists ? by_rank[t] : 0u;
        const uint32_t len_i = exists ? eff[row_i] : 0u;
        const int m = __popc(__ballot_sync(kFull, exists));
        const uint32_t vb = __ballot_sync(kFull, exists && len_i > 0 && lane < (int)csize);
        const int mv = __ffs(~vb) - 1;   // leading lanes with work
        // One CTA per row, then each spare CTA to the row with the largest
        // slice len / c (ties to the earlier row): a warp arg-max per spare.
        // len < 2^24 and c <= 16, so the cross products fit 32 bits.
        uint32_t c = lane < mv ? 1u : 0u;
        const uint32_t lw = lane < mv ? len_i : 0u;
        for (int used = mv; used < (int)csize && mv > 0; ++used) {
            uint32_t bl = lw, bc = c > 0 ? c : 1u;
            int bi = lane;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint32_t ol = __shfl_xor_sync(kFull, bl, o), oc = __shfl_xor_sync(kFull, bc, o);
                const int oi = __shfl_xor_sync(kFull, bi, o);
                if (ol * bc > bl * oc || (ol * bc == bl * oc && oi < bi)) {
                    bl = ol;
                    bc = oc;
                    bi = oi;
                }
            }
            if (lane == bi) ++c;
        }
        const uint32_t cs_incl = warp_incl_scan(c);
        const uint32_t start = cs_incl - c;
        const uint32_t own = __ballot_sync(kFull, c > 0 && crank >= start && crank < start + c);
        const int owner = own ? __ffs(own) - 1 : 0;
        const uint32_t o_row = __shfl_sync(kFull, row_i, owner);
        const uint32_t o_g0 = __shfl_sync(kFull, start, owner);
        const uint32_t o_gs = __shfl_sync(kFull, c, owner);
        if (lane == 0) {
            slot[0] = own ? o_row : 0xFFFFFFFFu;   // -1: no row with work for this CTA
            slot[1] = own ? o_g0 : 0u;
            slot[2] = own ? o_gs : 0u;
            // The cluster's first CTA pads the rows with nothing to select.
            slot[3] = (uint32_t)(m - mv);
        }
        if (lane >= mv && lane < m) slot[4 + lane - mv] = row_i;
    }
    __syncthreads();
    RowGroup g;
    g.row = (int)slot[0];
    g.g0 = slot[1];
    g.gsize = slot[2];
    g.start = g.row >= 0 ? (int32_t)starts[g.row] : 0;
    g.len = g.row >= 0 ? (int32_t)eff[g.row] : 0;
    if (crank == 0) {
        const int npad = (int)slot[3];
        for (int i = 0; i < npad; ++i) {
            const int rr = (int)slot[4 + i];
            int64_t len;
            const bool ok = row_window_ok(p, rr, len);
            if (!ok && tid == 0)
                atomicOr(&g_status, len >= (int64_t)TOPK_RAGGED_MAX_LEN ? TOPK_DEV_LEN_ENVELOPE
                                                                         : TOPK_DEV_BAD_WINDOW);
            pad_out(p.out_idx + (int64_t)rr * p.k, p.out_val ? p.out_val + (int64_t)rr * p.k : nullptr,
                    0, p.k);
        }
    }
    __syncthreads();
    return g;
}

// ------------------------------------------------------------------------- //
// The one-CTA-per-row kernel, for batches of many rows.  A row that fits the
// registers takes short_row; any other row (or a short row whose buckets are
// too skewed) takes the general path below: the row is streamed once into
// shared memory (what does not fit is re-read from L2), an MSB-first radix
// select of 11, 11 and 10 bits finds the exact k-th key T, the winners
// (key > T) are gathered and sorted, and the first r ties (key == T) are
// placed by index.
//
// Every pass over the slice walks the same contiguous per-warp segments, U
// quads per lane in flight, so per-warp counts taken in one pass give
// index-ordered positions in a later one.
// ------------------------------------------------------------------------- //
// Five CTAs per SM (48 registers, a few bytes spilled): five rows in flight
// per SM ran faster than four at 64 registers.
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 5) topk_row_kernel(const Params p)
{
    grid_dependency_enter();
    constexpr int NW = THREADS / 32;
    constexpr int U = 4;                       // quads in flight per lane
    constexpr uint32_t kZeroKey = 0x80000000u; // order key of +0.0
    constexpr uint32_t kZeroDigit = kZeroKey >> 21;
    extern __shared__ __align__(16) unsigned char smem[];
    Ctrl &ctrl = *reinterpret_cast<Ctrl *>(smem);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + sizeof(Ctrl));
    uint64_t *win = reinterpret_cast<uint64_t *>(smem + p.off_win);
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + p.off_keys);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Rows are dealt from the last one back: a causal prefill batch ends
    // with its longest rows, and taking those first shortens the tail.
    const int row = p.B - 1 - (int)blockIdx.x;

    // ---- a1: metadata, window checks ----------------------------------- //
    const int64_t rs = p.row_starts[row];
    int64_t len = p.lengths[row];
    // The row about one wave of CTAs later: its metadata loads along with
    // this row's, and its scores are prefetched into L2 below, so the CTA
    // that takes it later finds them there.
    int64_t rs_a = 0, len_a = 0;
    if (warp == THREADS / 32 - 1 && row - p.ahead >= 0 && p.ahead > 0) {
        rs_a = p.row_starts[row - p.ahead];
        len_a = p.lengths[row - p.ahead];
    }
    if (len < 0) len = 0;
    uint32_t bad = 0;
    if (len >= (int64_t)TOPK_RAGGED_MAX_LEN)
        bad = TOPK_DEV_LEN_ENVELOPE;
    else if (rs < 0 || rs + len > p.n_scores)
        bad = TOPK_DEV_BAD_WINDOW;
    int32_t *oi = p.out_idx + (int64_t)row * p.k;
    float *ov = p.out_val ? p.out_val + (int64_t)row * p.k : nullptr;
    if (bad || len == 0) {
        if (bad && tid == 0) atomicOr(&g_status, bad);
        pad_out(oi, ov, 0, p.k);
        return;
    }
    const int32_t L = (int32_t)len;
    const uint32_t k_eff = (uint32_t)(p.k < L ? p.k : L);
    const int64_t idx_offset = (p.offset_mode & TOPK_OFFSET_ROW_START) ? rs : 0;
    const bool excl = (p.offset_mode & TOPK_EXCLUDE_NEG_INF) != 0;

    // ---- slice of this CTA (16-byte aligned body split by quads) ----------- //
    Slice s;
    {
        // Slot 0 is the 16-byte aligned element at or before the row start.
        const int32_t mis = (int32_t)(((uintptr_t)(p.scores + rs) >> 2) & 3u);
        s.gptr = p.scores + (rs - mis);
        s.off0 = mis;
        s.end = mis + L;
        s.bq0 = mis ? 1 : 0;
        s.bq1 = max(s.bq0, s.end >> 2);
        s.nq = (s.end + 3) >> 2;
        s.sq = min(s.nq, p.stage_cap >> 2);
        s.jbase = -mis;
    }
    if (len_a > 0 && rs_a >= 0 && rs_a + len_a <= p.n_scores) {
        const char *b = reinterpret_cast<const char *>(p.scores + rs_a);
        const int64_t nbytes = min(len_a * 4, (int64_t)32768);
        for (int64_t o = (int64_t)lane * 128; o < nbytes; o += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(b + o));
    }
    if (s.nq <= kShortQuads * THREADS) {
        const uint32_t area = (uint32_t)(p.off_keys + p.stage_cap * 4) - (uint32_t)sizeof(Ctrl);
        if (short_row<THREADS>(ctrl, reinterpret_cast<unsigned char *>(hist), area, s, k_eff, idx_offset, oi, ov,
                               p.k, excl)) {
            if (p.page_table) {
                __syncthreads();
                page_map_row(p, row, oi, (int)k_eff);
            }
            return;
        }
    }
    const WarpSeg seg = warp_segment<THREADS>(s.nq, warp);

    // ---- init shared state ------------------------------------------------ //
    for (int b = tid; b < kBins; b += THREADS) hist[b] = 0u;
    if (tid == 0) {
        ctrl.sel_digit = 0u;
        ctrl.sel_gt = 0u;
        ctrl.sel_cnt = 0u;
        ctrl.sel_done = 0u;
        ctrl.zeros = 0u;
        ctrl.win_count = 0u;
        ctrl.kmax = 0u;
        ctrl.wmin = kFull;
    }
    __syncthreads();

    // ---- a2+a3: stream the slice once: key transform, stage, top-digit
    //      histogram, the largest key and per-warp counts of exact +0.0 --- //
    {
        uint32_t zeros = 0, kmax = 0;
        for (int qb = seg.q0; qb < seg.q1; qb += 32 * U) {
            uint4 kk[U];
            uint32_t m[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = qb + u * 32 + lane;
                m[u] = 0;
                kk[u] = make_uint4(0, 0, 0, 0);
                if (q < seg.q1) kk[u] = load_quad_global(s, q, m[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (qb + u * 32 >= seg.q1) break;   // warp-uniform
                const int q = qb + u * 32 + lane;
                if (q < s.sq && q < seg.q1) reinterpret_cast<uint4 *>(keys)[q] = kk[u];
                const uint32_t e[4] = {kk[u].x, kk[u].y, kk[u].z, kk[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bool v = (m[u] >> i) & 1u;
                    zeros += v && e[i] == kZeroKey;
                    kmax = max(kmax, v ? e[i] : 0u);
                    hist_add(hist, e[i] >> 21, v);
                }
            }
        }
        zeros = __reduce_add_sync(kFull, zeros);
        kmax = __reduce_max_sync(kFull, kmax);
        if (lane == 0) {
            ctrl.warp_zeros[warp] = zeros;
            if (zeros) atomicAdd(&ctrl.zeros, zeros);
            atomicMax(&ctrl.kmax, kmax);
        }
    }
    __syncthreads();

    // Running selection state (identical in every thread).
    uint32_t prefix = 0, n_gt = 0, r = k_eff, cnt = 0;
    bool plateau = false;   // T is +0.0, found from the zero count
    bool sel_done = false;  // the k-th key is known

    // ---- a4+a5: radix levels of 11, 11 and 10 bits --------------------- //
#pragma unroll 1
    for (int level = 0; level < 3; ++level) {
        const int dbits = level == 2 ? 10 : 11;
        if (level > 0 && !sel_done) {
            const int pshift = level == 1 ? 21 : 10;
            const int dshift = level == 1 ? 10 : 0;
            const uint32_t dmask = (1u << dbits) - 1u;
            for (int qb = seg.q0; qb < seg.q1; qb += 32 * U) {
                uint4 kk[U];
                uint32_t m[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int q = qb + u * 32 + lane;
                    m[u] = 0;
                    kk[u] = make_uint4(0, 0, 0, 0);
                    if (q < seg.q1) kk[u] = load_quad(s, keys, q, m[u]);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (qb + u * 32 >= seg.q1) break;   // warp-uniform
                    const uint32_t e[4] = {kk[u].x, kk[u].y, kk[u].z, kk[u].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const bool v = ((m[u] >> i) & 1u) && (e[i] >> pshift) == prefix;
                        hist_add(hist, (e[i] >> dshift) & dmask, v);
                    }
                }
            }
            __syncthreads();
        }
        uint32_t d = 0, gt = 0, c = 0;
        if (!sel_done) {
            if (find_bin<THREADS>(hist, r, ctrl.scan, d, gt, c)) {
                // Plateau shortcut: the boundary bin holds only exact +0.0, so
                // the k-th key is +0.0 and the finer levels are not needed.
                ctrl.sel_digit = d;
                ctrl.sel_gt = gt;
                ctrl.sel_cnt = c;
                ctrl.sel_done = (level == 0 && d == kZeroDigit && c == ctrl.zeros) ? 1u : 0u;
            }
        }
        __syncthreads();
        if (!sel_done) {
            d = ctrl.sel_digit;
            gt = ctrl.sel_gt;
            c = ctrl.sel_cnt;
            const bool done = ctrl.sel_done != 0u;
            // Exact integer counts guarantee gt < r <= gt + c; anything else
            // is a library bug: flag it and keep every later write in the row.
            if (gt >= r || r - gt > c) {
                if (tid == 0) atomicOr(&g_status, TOPK_DEV_INTERNAL);
                gt = r - 1u;
                c = 1u;
            }
            n_gt += gt;
            r -= gt;
            cnt = c;
            if (done) {
                prefix = kZeroKey;
                plateau = true;
                sel_done = true;
            } else {
                prefix = (prefix << dbits) | d;
                if (level == 2) sel_done = true;
                else
                    for (int b = tid; b < kBins; b += THREADS) hist[b] = 0u;
            }
        }
        __syncthreads();
        if (sel_done) break;
    }
    const uint32_t T = prefix;   // exact k-th key; n_gt above it, take r of its cnt ties

    // ---- a6+a7: one pass over the slice.  Winners (key > T) go to the
    //      list in any order (their composites are unique, the sort makes
    //      the order canonical).  Ties (key == T): the first r in index
    //      order go straight to positions n_gt + ordinal.  On the plateau
    //      every tie is a +0.0 and the per-warp zero counts of the streaming
    //      pass already give each warp's first ordinal; else the pass counts
    //      ties per warp and a second pass writes them. ------------------- //
    const uint32_t tie_base = 0, local_eq = cnt;
    const bool want_ties = local_eq > 0 && tie_base < r;   // CTA-uniform
    uint32_t trun = 0;   // this warp's next tie ordinal (plateau)
    if (plateau && want_ties) {
        if (warp == 0) {
            const uint32_t z = lane < NW ? ctrl.warp_zeros[lane] : 0u;
            const uint32_t zi = warp_incl_scan(z);
            if (lane < NW) ctrl.warp_ties[lane] = zi - z;
        }
        __syncthreads();
        trun = tie_base + ctrl.warp_ties[warp];
    }
    const bool fused_ties = plateau && want_ties && ctrl.warp_zeros[warp] > 0;   // warp-uniform
    uint32_t ties_w = 0, wmin = kFull;
    int first_tie_q = seg.q1;
    const uint32_t lt = lanemask_lt();
    for (int qb = seg.q0; qb < seg.q1; qb += 32 * U) {
        uint4 kk[U];
        uint32_t m[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = qb + u * 32 + lane;
            m[u] = 0;
            kk[u] = make_uint4(0, 0, 0, 0);
            if (q < seg.q1) kk[u] = load_quad(s, keys, q, m[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (qb + u * 32 >= seg.q1) break;   // warp-uniform
            const int q = qb + u * 32 + lane;
            const uint32_t e[4] = {kk[u].x, kk[u].y, kk[u].z, kk[u].w};
            uint32_t wm = 0, tm = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if ((m[u] >> i) & 1u) {
                    if (e[i] > T) wm |= 1u << i;
                    else if (e[i] == T) tm |= 1u << i;
                }
            }
            // Per-slot ballots give every lane its prefix count without a
            // shuffle scan; lane order then slot order is index order.
            if (__ballot_sync(kFull, wm != 0)) {
                uint32_t wtot = 0, slot = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t b = __ballot_sync(kFull, (wm >> i) & 1u);
                    wtot += (uint32_t)__popc(b);
                    slot += (uint32_t)__popc(b & lt);
                }
                uint32_t base = 0;
                if (lane == 0)
                    base = atomicAdd(&ctrl.win_count, wtot);
                slot += __shfl_sync(kFull, base, 0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if ((wm >> i) & 1u) {
                        const uint32_t j = (uint32_t)(s.jbase + 4 * q + i);
                        const uint64_t comp = ((uint64_t)e[i] << 32) | (uint64_t)(~j);
                        wmin = min(wmin, e[i]);
                        if (slot < (uint32_t)p.win_cap) win[slot] = comp;
                        ++slot;
                    }
                }
            }
            const uint32_t tany = __ballot_sync(kFull, tm != 0);
            if (tany) {
                uint32_t ttot = 0, tord = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t b = __ballot_sync(kFull, (tm >> i) & 1u);
                    ttot += (uint32_t)__popc(b);
                    tord += (uint32_t)__popc(b & lt);
                }
                if (fused_ties) {
                    if (trun < r) {
                        tord += trun;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            if ((tm >> i) & 1u) {
                                if (tord < r && n_gt + tord < k_eff) {
                                    const int32_t j = s.jbase + 4 * q + i;
                                    put_out(oi, ov, n_gt + tord, idx_offset, j, T, excl);
                                }
                                ++tord;
                            }
                        }
                    }
                    trun += ttot;
                } else if (want_ties) {
                    ties_w += ttot;
                    const int fq = qb + u * 32 + __ffs(tany) - 1;
                    if (fq < first_tie_q) first_tie_q = fq;
                }
            }
        }
    }
    wmin = __reduce_min_sync(kFull, wmin);
    if (lane == 0 && wmin != kFull) atomicMin(&ctrl.wmin, wmin);

    // ---- a7 (off the plateau): ties in index order, per-warp bases from
    //      the counts above; each warp starts at its first tie ------------ //
    if (want_ties && !plateau) {
        if (lane == 0) ctrl.warp_ties[warp] = ties_w;
        __syncthreads();
        if (warp == 0) {
            const uint32_t b = lane < NW ? ctrl.warp_ties[lane] : 0u;
            const uint32_t bi = warp_incl_scan(b);
            if (lane < NW) ctrl.warp_ties[lane] = bi - b;
        }
        __syncthreads();
        trun = tie_base + ctrl.warp_ties[warp];
        if (ties_w > 0 && trun < r) {   // warp-uniform
            for (int qb = first_tie_q; qb < seg.q1 && trun < r; qb += 32) {
                const int q = qb + lane;
                uint32_t m = 0;
                uint4 kk = make_uint4(0, 0, 0, 0);
                if (q < seg.q1) kk = load_quad(s, keys, q, m);
                const uint32_t e[4] = {kk.x, kk.y, kk.z, kk.w};
                uint32_t tm = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (((m >> i) & 1u) && e[i] == T) tm |= 1u << i;
                if (__ballot_sync(kFull, tm != 0)) {
                    uint32_t ttot = 0, tord = trun;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t b = __ballot_sync(kFull, (tm >> i) & 1u);
                        ttot += (uint32_t)__popc(b);
                        tord += (uint32_t)__popc(b & lt);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if ((tm >> i) & 1u) {
                            if (tord < r && n_gt + tord < k_eff) {
                                const int32_t j = s.jbase + 4 * q + i;
                                put_out(oi, ov, n_gt + tord, idx_offset, j, T, excl);
                            }
                            ++tord;
                        }
                    }
                    trun += ttot;
                }
            }
        }
    }

    // ---- a8+a9: sort the winners and write the row ---------------------- //
    __syncthreads();
    const uint32_t n_win = ctrl.win_count;
    if (n_win != n_gt || n_gt > (uint32_t)p.win_cap) {
        if (tid == 0) atomicOr(&g_status, TOPK_DEV_INTERNAL);
    }
    const uint32_t n_sort = n_gt < (uint32_t)p.win_cap ? n_gt : (uint32_t)p.win_cap;
    if (n_sort > 0) {
        sort_and_write<THREADS>(win, reinterpret_cast<uint64_t *>(keys), (int)n_sort, (int)n_sort, p.win_cap,
                                ctrl.wmin, ctrl.kmax, hist, ctrl.scan64, oi, ov, idx_offset, excl);
    }
    pad_out(oi, ov, (int)k_eff, p.k);
    if (p.page_table) {
        __syncthreads();
        page_map_row(p, row, oi, (int)k_eff);
    }
}

// ------------------------------------------------------------------------- //
// The cluster kernel: each cluster of CS CTAs takes a group of rows
// (assign_rows) and every row is worked on by a contiguous group of the
// cluster's CTAs; the group's first CTA is the row's leader, which sorts the
// row's candidates and writes it.
//
//   1. Each CTA starts bulk copies (TMA) of its whole staged slice into
//      shared memory, so every byte of the batch is in flight at once.
//   2. Level 0: one pass over the slice turns scores into order keys in
//      place and builds the 11-bit top-digit histogram.  After a cluster
//      barrier every CTA of the group pulls its peers' histograms over DSMEM
//      and runs the same threshold search, so all of them hold the same
//      exact integers without a round trip through the leader.
//   3. The row then either
//        * is on the +0.0 plateau (the boundary bin holds only +0.0), or
//        * has few enough entries at or above the boundary bin to sort
//          them all (candidates: every key >= the bin's lower bound), or
//        * refines the boundary bin by the next 11 bits (level 1) and,
//          if still too many, the last 10 bits (level 2), which gives the
//          exact k-th key T.
//      The histograms of consecutive levels live in different buffers,
//      so one cluster barrier per level is enough.
//   4. Compaction: candidates go to the CTA's own list.  With an exact T
//      the entries equal to T are ties: the first r of them in index order
//      go straight to output positions n_gt + ordinal.
//   5. After the last level barrier the leader pulls the group's lists into
//      its staging area over DSMEM, releases the peers (a split cluster
//      barrier) and sorts the candidates and writes the row.
// Every CTA of the cluster runs the same four cluster barriers whatever
// its row needs.
// ------------------------------------------------------------------------- //

// Sum of the group's histograms over this thread's BPT bins starting at lo.
template <int THREADS>
__device__ __forceinline__ void pull_bins(const uint32_t *h, int lo, uint32_t g0, uint32_t gsize, uint32_t crank,
                                          uint32_t (&v)[kBins / THREADS])
{
    constexpr int BPT = kBins / THREADS;
    constexpr int kBatch = 4;   // remote loads in flight before they are summed
    load_bins<THREADS>(h, lo, v);
    for (uint32_t r0 = g0; r0 < g0 + gsize; r0 += kBatch) {
        uint32_t w[kBatch][BPT];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const uint32_t r = r0 + (uint32_t)b;
            if (r < g0 + gsize && r != crank) {
                dsmem_ld_bins(dsmem_addr(h + lo, r), w[b]);
            } else {
#pragma unroll
                for (int i = 0; i < BPT; ++i) w[b][i] = 0u;
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
#pragma unroll
            for (int i = 0; i < BPT; ++i) v[i] += w[b][i];
    }
}

// Threshold search on bins already in registers (see find_bin).
template <int THREADS>
__device__ __forceinline__ bool find_bin_v(const uint32_t (&v)[kBins / THREADS], int lo, uint32_t r, uint32_t *sm,
                                           uint32_t &digit, uint32_t &gt, uint32_t &cnt)
{
    constexpr int BPT = kBins / THREADS;
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) sum += v[i];
    const uint32_t incl = block_incl_scan<THREADS>(sum, sm);
    const uint32_t excl = incl - sum;
    bool mine = false;
    if (excl < r && r <= incl) {
        uint32_t acc = excl;
#pragma unroll
        for (int i = BPT - 1; i >= 0; --i) {
            if (!mine && acc + v[i] >= r) {
                mine = true;
                digit = (uint32_t)(lo + i);
                gt = acc;
                cnt = v[i];
            }
            acc += v[i];
        }
    }
    return mine;
}

// Pulls the group's histogram h, finds the bin holding the r-th largest
// entry and returns (digit, entries above it, entries in it) to every
// thread.  Ends with a __syncthreads.
template <int THREADS>
__device__ __forceinline__ void group_select(CCtrl &ctrl, const uint32_t *h, uint32_t g0, uint32_t gsize,
                                             uint32_t crank, uint32_t r, uint32_t &d, uint32_t &gt, uint32_t &c)
{
    constexpr int BPT = kBins / THREADS;
    const int lo = kBins - ((int)threadIdx.x + 1) * BPT;   // thread 0 owns the top bins
    uint32_t v[BPT];
    pull_bins<THREADS>(h, lo, g0, gsize, crank, v);
    uint32_t dd, gg, cc;
    if (find_bin_v<THREADS>(v, lo, r, ctrl.scan, dd, gg, cc)) {
        ctrl.sel[0] = dd;
        ctrl.sel[1] = gg;
        ctrl.sel[2] = cc;
    }
    __syncthreads();
    d = ctrl.sel[0];
    gt = ctrl.sel[1];
    c = ctrl.sel[2];
}

// The slice's quads in index order: an optional partial head quad (0), the
// full quads [bq0, bq1) cut into one contiguous run per warp, and an
// optional partial tail quad (nq - 1).  Warp 0 owns the head and the last
// warp the tail, so warp order is index order and the inner loops need no
// per-slot masks.
// Quads per lane in flight in the cluster kernel's passes.
constexpr int kPassQuads = 2;

struct Parts {
    int q0, q1;       // this warp's run of full quads
    int head, tail;   // partial quads this warp owns, or -1
};

template <int THREADS>
__device__ __forceinline__ Parts slice_parts(const Slice &s, int warp)
{
    constexpr int NW = THREADS / 32;
    Parts pt;
    const int n = s.bq1 - s.bq0;
    const int per = (n + NW - 1) / NW;
    pt.q0 = s.bq0 + min(n, warp * per);
    pt.q1 = s.bq0 + min(n, warp * per + per);
    const int head = s.bq0 > 0 ? 0 : -1;
    const int tail = (s.nq > s.bq1 && s.nq - 1 != head) ? s.nq - 1 : -1;
    pt.head = warp == 0 ? head : -1;
    pt.tail = warp == NW - 1 ? tail : -1;
    return pt;
}

// A fully staged slice (every quad in shared memory) whose partial end
// quads hold the sentinel key 0 in their empty slots: every warp takes a
// contiguous run of all nq quads and there are no separate partial quads.
// Level 0 counts the sentinels into bin 0 and takes them out again; the
// later passes use it only when their key range excludes 0.
template <int THREADS>
__device__ __forceinline__ Parts staged_parts(const Slice &s, int warp)
{
    const WarpSeg w = warp_segment<THREADS>(s.nq, warp);
    Parts pt;
    pt.q0 = w.q0;
    pt.q1 = w.q1;
    pt.head = -1;
    pt.tail = -1;
    return pt;
}

__device__ __forceinline__ uint4 to_keys(uint4 raw)
{
    return make_uint4(order_key(raw.x), order_key(raw.y), order_key(raw.z), order_key(raw.w));
}

// A full quad's keys: staged (already keys) or read from global memory.
__device__ __forceinline__ uint4 body_quad(const Slice &s, const uint4 *keys4, int q)
{
    if (q < s.sq) return keys4[q];
    const float4 f = __ldg(reinterpret_cast<const float4 *>(s.gptr) + q);
    return make_uint4(order_key(__float_as_uint(f.x)), order_key(__float_as_uint(f.y)),
                      order_key(__float_as_uint(f.z)), order_key(__float_as_uint(f.w)));
}

// Runs f(kk, valid) over this warp's full quads, U per lane a round; valid
// says whether the lane's quad u exists.  STAGED: every quad is in shared
// memory.
template <int U, bool STAGED, class F>
__device__ __forceinline__ void body_rounds(const Slice &s, const uint4 *keys4, const Parts &pt, F &&f)
{
    const int lane = threadIdx.x & 31;
    for (int qb = pt.q0; qb < pt.q1; qb += 32 * U) {
        uint4 kk[U];
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = qb + u * 32 + lane;
            ok[u] = q < pt.q1;
            kk[u] = make_uint4(0, 0, 0, 0);
            if (ok[u]) kk[u] = STAGED ? keys4[q] : body_quad(s, keys4, q);
        }
        f(qb, kk, ok);
    }
}

// Level-0 pass: staged scores become keys in place; entries are counted by
// their top 11 bits, exact +0.0 per warp (about half of a ReLU row) rather
// than by atomics on one bin.
template <int THREADS, bool STAGED>
__device__ void level0_pass(CCtrl &ctrl, const Slice &s, uint32_t *keys, const Parts &pt, uint32_t *hist,
                            uint32_t n_sentinel)
{
    constexpr int U = kPassQuads;
    constexpr uint32_t kZ = 0x80000000u;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint4 *keys4 = reinterpret_cast<uint4 *>(keys);
    uint32_t zeros = 0;
    auto take = [&](uint32_t e, bool v) {
        const bool z = e == kZ;
        zeros += v && z;
        if (v && !z) hist_inc(hist, e >> 21);
    };
    for (int qb = pt.q0; qb < pt.q1; qb += 32 * U) {
        uint4 kk[U];
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = qb + u * 32 + lane;
            ok[u] = q < pt.q1;
            kk[u] = make_uint4(0, 0, 0, 0);
            if (ok[u]) {
                if (STAGED || q < s.sq) {
                    kk[u] = to_keys(keys4[q]);
                    keys4[q] = kk[u];
                } else {
                    kk[u] = body_quad(s, keys4, q);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            take(kk[u].x, ok[u]);
            take(kk[u].y, ok[u]);
            take(kk[u].z, ok[u]);
            take(kk[u].w, ok[u]);
        }
    }
    if (lane == 0) {
        for (int h = 0; h < 2; ++h) {
            const int q = h == 0 ? pt.head : pt.tail;
            if (q < 0) continue;
            uint32_t m;
            uint4 kk;
            if (q < s.sq) {
                m = quad_mask(s, q);
                kk = to_keys(keys4[q]);
                keys4[q] = kk;
            } else {
                kk = load_quad_global(s, q, m);
            }
            take(kk.x, m & 1u);
            take(kk.y, (m >> 1) & 1u);
            take(kk.z, (m >> 2) & 1u);
            take(kk.w, (m >> 3) & 1u);
        }
    }
    zeros = __reduce_add_sync(kFull, zeros);
    if (lane == 0) {
        ctrl.warp_zeros[warp] = zeros;
        if (zeros) {
            atomicAdd(&ctrl.zeros, zeros);
            atomicAdd(&hist[kZ >> 21], zeros);
        }
    }
    if (STAGED && threadIdx.x == 0 && n_sentinel) atomicSub(&hist[0], n_sentinel);
}

// A partial quad's keys (after level 0) and its valid slots.
__device__ __forceinline__ uint4 partial_quad(const Slice &s, const uint4 *keys4, int q, uint32_t &m)
{
    if (q < s.sq) {
        m = quad_mask(s, q);
        return keys4[q];
    }
    return load_quad_global(s, q, m);
}

__device__ __forceinline__ uint32_t quad_max(const uint4 &k)
{
    return max(max(k.x, k.y), max(k.z, k.w));
}

__device__ __forceinline__ uint32_t quad_min(const uint4 &k)
{
    return min(min(k.x, k.y), min(k.z, k.w));
}

// Refinement pass: entries whose key matches `prefix` above bit `pshift`
// (a key range [plo, phi]) are counted by the digit (key >> dshift) & dmask.
// A quad is looked at entry by entry only when its range meets [plo, phi].
template <int THREADS, bool STAGED>
__device__ void level_pass(const Slice &s, const uint32_t *keys, const Parts &pt, uint32_t *hist, uint32_t prefix,
                           int pshift, int dshift, uint32_t dmask)
{
    constexpr int U = kPassQuads;
    const uint4 *keys4 = reinterpret_cast<const uint4 *>(keys);
    const uint32_t plo = prefix << pshift, phi = plo | ((1u << pshift) - 1u);
    auto take = [&](uint32_t e, bool v) {
        if (v && e >= plo && e <= phi) hist_inc(hist, (e >> dshift) & dmask);
    };
    body_rounds<U, STAGED>(s, keys4, pt, [&](int, const uint4 (&kk)[U], const bool (&ok)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (ok[u] && quad_max(kk[u]) >= plo && quad_min(kk[u]) <= phi) {
                take(kk[u].x, true);
                take(kk[u].y, true);
                take(kk[u].z, true);
                take(kk[u].w, true);
            }
        }
    });
    if ((threadIdx.x & 31) == 0) {
        for (int h = 0; h < 2; ++h) {
            const int q = h == 0 ? pt.head : pt.tail;
            if (q < 0) continue;
            uint32_t m;
            const uint4 kk = partial_quad(s, keys4, q, m);
            take(kk.x, m & 1u);
            take(kk.y, (m >> 1) & 1u);
            take(kk.z, (m >> 2) & 1u);
            take(kk.w, (m >> 3) & 1u);
        }
    }
}

// Compaction.  Candidates (EXACT: key > T; else key >= lo) go to this CTA's
// own list; with an exact T the ties (key == T) take output positions
// n_gt + ordinal for ordinals below r, in group-wide index order starting at
// tie_base.  A count pass gives every warp its base in the list and in the
// tie order, and a write pass places the entries with warp scans, so the
// list comes out in index order with no shared counter.  The smallest and
// largest candidate keys go to ctrl.wmin / ctrl.wmax.  Ends with a
// __syncthreads; the list length is left in ctrl.win_local.
template <int THREADS, bool EXACT, bool STAGED>
__device__ void compact_slice(CCtrl &ctrl, const Slice &s, const uint32_t *keys, const Parts &pt, uint64_t *win,
                              uint32_t wcap, uint32_t lo, uint32_t T, uint32_t tie_base, uint32_t r, uint32_t n_gt,
                              uint32_t k_eff, int64_t idx_offset, int32_t *oi, float *ov, bool excl)
{
    constexpr int NW = THREADS / 32;
    constexpr int U = kPassQuads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4 *keys4 = reinterpret_cast<const uint4 *>(keys);
    auto is_cand = [&](uint32_t e) { return EXACT ? e > T : e >= lo; };
    auto is_tie = [&](uint32_t e) { return EXACT && e == T; };

    if constexpr (!EXACT) {
        // Without ties the list's order is free: one pass, each warp round
        // taking its slots with one atomic on the list length.
        if (tid == 0) ctrl.win_local = 0u;
        __syncthreads();
        uint32_t wmin = kFull, wmax = 0;
        auto put = [&](uint32_t e, int32_t j, uint32_t slot) {
            wmin = min(wmin, e);
            wmax = max(wmax, e);
            if (slot < wcap) win[slot] = ((uint64_t)e << 32) | (uint64_t)(~(uint32_t)j);
        };
        if (pt.head >= 0 || pt.tail >= 0) {   // warp-uniform
            for (int h = 0; h < 2; ++h) {
                const int q = h == 0 ? pt.head : pt.tail;
                if (q < 0) continue;
                uint32_t c = 0, m = 0;
                uint4 kk = make_uint4(0, 0, 0, 0);
                if (lane == 0) {
                    kk = partial_quad(s, keys4, q, m);
                    const uint32_t e[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) c += ((m >> i) & 1u) && e[i] >= lo;
                }
                uint32_t base = 0;
                if (lane == 0 && c) base = atomicAdd(&ctrl.win_local, c);
                if (lane == 0 && c) {
                    const uint32_t e[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (((m >> i) & 1u) && e[i] >= lo) put(e[i], s.jbase + 4 * q + i, base++);
                }
            }
        }
        body_rounds<U, STAGED>(s, keys4, pt, [&](int qb, const uint4 (&kk)[U], const bool (&ok)[U]) {
            uint32_t cm = 0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!(ok[u] && quad_max(kk[u]) >= lo)) continue;
                const uint32_t e[4] = {kk[u].x, kk[u].y, kk[u].z, kk[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) cm |= (uint32_t)(e[i] >= lo) << (4 * u + i);
            }
            if (!__any_sync(kFull, cm != 0)) return;
            const uint32_t cnt = (uint32_t)__popc(cm);
            const uint32_t ci = warp_incl_scan(cnt);
            uint32_t base = 0;
            if (lane == 31) base = atomicAdd(&ctrl.win_local, ci);
            uint32_t slot = __shfl_sync(kFull, base, 31) + ci - cnt;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t e[4] = {kk[u].x, kk[u].y, kk[u].z, kk[u].w};
                const int32_t j0 = s.jbase + 4 * (qb + u * 32 + lane);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if ((cm >> (4 * u + i)) & 1u) put(e[i], j0 + i, slot++);
            }
        });
        wmin = __reduce_min_sync(kFull, wmin);
        wmax = __reduce_max_sync(kFull, wmax);
        if (lane == 0 && wmin != kFull) {
            atomicMin(&ctrl.wmin, wmin);
            atomicMax(&ctrl.wmax, wmax);
        }
        __syncthreads();
        return;
    }

    // Count pass.
    uint32_t nc = 0, nt = 0;
    auto count = [&](uint32_t e, bool v) {
        nc += v && is_cand(e);
        nt += v && is_tie(e);
    };
    // Candidates and ties are both >= thr: most quads are passed over on
    // their largest key.
    const uint32_t thr = EXACT ? T : lo;
    body_rounds<U, STAGED>(s, keys4, pt, [&](int, const uint4 (&kk)[U], const bool (&ok)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (ok[u] && quad_max(kk[u]) >= thr) {
                count(kk[u].x, true);
                count(kk[u].y, true);
                count(kk[u].z, true);
                count(kk[u].w, true);
            }
        }
    });
    if (lane == 0) {
        for (int h = 0; h < 2; ++h) {
            const int q = h == 0 ? pt.head : pt.tail;
            if (q < 0) continue;
            uint32_t m;
            const uint4 kk = partial_quad(s, keys4, q, m);
            count(kk.x, m & 1u);
            count(kk.y, (m >> 1) & 1u);
            count(kk.z, (m >> 2) & 1u);
            count(kk.w, (m >> 3) & 1u);
        }
    }
    nc = __reduce_add_sync(kFull, nc);
    nt = __reduce_add_sync(kFull, nt);
    if (lane == 0) {
        ctrl.warp_zeros[warp] = nc;
        ctrl.warp_ties[warp] = nt;
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t c = lane < NW ? ctrl.warp_zeros[lane] : 0u;
        const uint32_t t = lane < NW ? ctrl.warp_ties[lane] : 0u;
        const uint32_t ci = warp_incl_scan(c), ti = warp_incl_scan(t);
        if (lane < NW) {
            ctrl.warp_zeros[lane] = ci - c;
            ctrl.warp_ties[lane] = ti - t;
        }
        if (lane == 31) ctrl.win_local = ci;
    }
    __syncthreads();

    // Write pass.
    uint32_t cbase = ctrl.warp_zeros[warp], tbase = tie_base + ctrl.warp_ties[warp];
    uint32_t wmin = kFull, wmax = 0;
    auto put_cand = [&](uint32_t e, int32_t j, uint32_t slot) {
        wmin = min(wmin, e);
        wmax = max(wmax, e);
        if (slot < wcap) win[slot] = ((uint64_t)e << 32) | (uint64_t)(~(uint32_t)j);
    };
    auto put_tie = [&](int32_t j, uint32_t ord) {
        if (ord < r && n_gt + ord < k_eff) put_out(oi, ov, n_gt + ord, idx_offset, j, T, excl);
    };
    // A partial quad of this warp, written by lane 0 at the warp's cursors.
    auto partial = [&](int q) {
        uint32_t c = 0, t = 0;
        if (lane == 0) {
            uint32_t m;
            const uint4 kk = partial_quad(s, keys4, q, m);
            const uint32_t e[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (!((m >> i) & 1u)) continue;
                if (is_cand(e[i])) put_cand(e[i], s.jbase + 4 * q + i, cbase + c++);
                if (is_tie(e[i])) put_tie(s.jbase + 4 * q + i, tbase + t++);
            }
        }
        cbase += __shfl_sync(kFull, c, 0);
        tbase += __shfl_sync(kFull, t, 0);
    };
    if (nc > 0 || (nt > 0 && tbase < r)) {   // warp-uniform
        if (pt.head >= 0) partial(pt.head);
        body_rounds<U, STAGED>(s, keys4, pt, [&](int qb, const uint4 (&kk)[U], const bool (&ok)[U]) {
            uint32_t cm = 0, tm = 0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!(ok[u] && quad_max(kk[u]) >= thr)) continue;
                const uint32_t e[4] = {kk[u].x, kk[u].y, kk[u].z, kk[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    cm |= (uint32_t)is_cand(e[i]) << (4 * u + i);
                    if (EXACT) tm |= (uint32_t)is_tie(e[i]) << (4 * u + i);
                }
            }
            if (__any_sync(kFull, cm != 0)) {
                // Candidates: slots by a lane prefix (their order is free).
                const uint32_t cnt = (uint32_t)__popc(cm);
                const uint32_t ci = warp_incl_scan(cnt);
                uint32_t slot = cbase + ci - cnt;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t e[4] = {kk[u].x, kk[u].y, kk[u].z, kk[u].w};
                    const int32_t j0 = s.jbase + 4 * (qb + u * 32 + lane);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if ((cm >> (4 * u + i)) & 1u) put_cand(e[i], j0 + i, slot++);
                }
                cbase += __shfl_sync(kFull, ci, 31);
            }
            if (EXACT && __any_sync(kFull, tm != 0)) {
                // Ties follow index order, which within a round is quad u,
                // then lane, then slot: counts per u packed a byte each
                // (at most 128) into one warp scan.
                uint32_t packed = 0;
#pragma unroll
                for (int u = 0; u < U; ++u) packed |= (uint32_t)__popc((tm >> (4 * u)) & 0xFu) << (8 * u);
                const uint32_t ti = warp_incl_scan(packed);
                const uint32_t ttot = __shfl_sync(kFull, ti, 31), tex = ti - packed;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    uint32_t ord = tbase + ((tex >> (8 * u)) & 0xFFu);
                    const int32_t j0 = s.jbase + 4 * (qb + u * 32 + lane);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if ((tm >> (4 * u + i)) & 1u) put_tie(j0 + i, ord++);
                    tbase += (ttot >> (8 * u)) & 0xFFu;
                }
            }
        });
        if (pt.tail >= 0) partial(pt.tail);
    }
    wmin = __reduce_min_sync(kFull, wmin);
    wmax = __reduce_max_sync(kFull, wmax);
    if (lane == 0 && wmin != kFull) {
        atomicMin(&ctrl.wmin, wmin);
        atomicMax(&ctrl.wmax, wmax);
    }
    __syncthreads();
}

__device__ __forceinline__ uint64_t dsmem_ld64(uint32_t addr)
{
    uint64_t v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}

// The staged (mask-free) passes serve when their key range excludes the
// sentinel key 0; otherwise, or for a slice not wholly staged, the masked
// passes run on the slice's own parts.
template <int THREADS>
__device__ __forceinline__ void refine_pass(bool staged, const Slice &s, const uint32_t *keys, const Parts &pt,
                                            const Parts &ptm, uint32_t *hist, uint32_t prefix, int pshift, int dshift,
                                            uint32_t dmask)
{
    if (staged && prefix != 0u) level_pass<THREADS, true>(s, keys, pt, hist, prefix, pshift, dshift, dmask);
    else level_pass<THREADS, false>(s, keys, ptm, hist, prefix, pshift, dshift, dmask);
}

template <int THREADS, bool EXACT>
__device__ __forceinline__ void compact(bool staged, CCtrl &ctrl, const Slice &s, const uint32_t *keys,
                                        const Parts &pt, const Parts &ptm, uint64_t *win, uint32_t wcap, uint32_t lo,
                                        uint32_t T, uint32_t tie_base, uint32_t r, uint32_t n_gt, uint32_t k_eff,
                                        int64_t idx_offset, int32_t *oi, float *ov, bool excl)
{
    if (staged && (EXACT ? T != 0u : lo != 0u))
        compact_slice<THREADS, EXACT, true>(ctrl, s, keys, pt, win, wcap, lo, T, tie_base, r, n_gt, k_eff, idx_offset,
                                            oi, ov, excl);
    else
        compact_slice<THREADS, EXACT, false>(ctrl, s, keys, ptm, win, wcap, lo, T, tie_base, r, n_gt, k_eff,
                                             idx_offset, oi, ov, excl);
}

// ------------------------------------------------------------------------- //
// Sampled path of the cluster kernel.
//
// Before the row's scores land in shared memory, every CTA of the row's
// group reads the same deterministic sample of the row (the whole row when
// L <= 4096, else 128 runs of 32 consecutive scores spread evenly over it)
// and takes from it a lower bound
// `lo` that, with overwhelming probability, lies at or below the k-th key:
// the sample's m-th largest key rounded down to its 11-bit digit, where m is
// the expected number of sampled entries above the k-th key plus four
// standard deviations and 8 (m = k exactly when the sample is the whole
// row).  One pass over the staged slice then keeps only the keys >= lo: they
// are counted in a fine histogram of kFineBins bins over [lo, ...) and
// appended to the CTA's candidate list as unique composites.  After one
// cluster barrier every CTA of the group sums the group's fine histograms,
// and the exclusive counts from the top give every fine bin its first output
// place.  Each CTA then takes the bins whose first place falls in its share
// of the output, gathers their members from the group's lists, ranks each
// member inside its bin (composites are unique) and writes it at its place.
// When the bound lies on or below the +0.0 key (a row whose k-th key may be
// on the ReLU plateau) the candidates are the positive keys and the +0.0
// entries are counted per warp: if the positives are fewer than k, the k-th
// key is +0.0 and the first k - |positives| of them in index order follow.
//
// Every decision is taken from exact integer counts that all CTAs of the
// group hold alike.  When a check fails (the bound was above the k-th key, a
// list overflowed, a bin holds too many members to rank cheaply, or the k-th
// key is below +0.0) the group falls back to the full radix select below,
// on the same staged slice, so the result is the same either way.
// ------------------------------------------------------------------------- //
constexpr int kSample = 4096;       // scores of a row's sample
constexpr int kFineBins = 1024;     // bins of the candidates' histogram
constexpr uint32_t kMaxFineBin = 256;   // members a fine bin may hold on the sampled path

// Fine bin of a candidate key e: bins of 2^sh keys from lo (the smallest
// sampled candidate key); keys below lo share bin 0, keys past the last bin
// share it.
__device__ __forceinline__ uint32_t fine_bin(uint32_t e, uint32_t lo, uint32_t sh)
{
    if (e < lo) return 0u;
    const uint32_t f = (e - lo) >> sh;
    return f < (uint32_t)kFineBins ? f : (uint32_t)kFineBins - 1u;
}

// A full quad of the slice as keys: staged quads hold raw score bits.
__device__ __forceinline__ uint4 raw_body_keys(const Slice &s, const uint4 *raw4, int q)
{
    if (q < s.sq) return to_keys(raw4[q]);
    const float4 f = __ldg(reinterpret_cast<const float4 *>(s.gptr) + q);
    return make_uint4(order_key(__float_as_uint(f.x)), order_key(__float_as_uint(f.y)),
                      order_key(__float_as_uint(f.z)), order_key(__float_as_uint(f.w)));
}

// A partial (head or tail) quad as keys, with its valid slots in m.
__device__ __forceinline__ uint4 raw_partial_keys(const Slice &s, const uint4 *raw4, int q, uint32_t &m)
{
    if (q < s.sq) {
        m = quad_mask(s, q);
        return to_keys(raw4[q]);
    }
    return load_quad_global(s, q, m);
}

// A full quad of the slice as raw score bits (staged, or read where it lies).
__device__ __forceinline__ uint4 raw_body_quad(const Slice &s, const uint4 *raw4, int q)
{
    if (q < s.sq) return raw4[q];
    const float4 f = __ldg(reinterpret_cast<const float4 *>(s.gptr) + q);
    return make_uint4(__float_as_uint(f.x), __float_as_uint(f.y), __float_as_uint(f.z), __float_as_uint(f.w));
}

// Appends a lane's candidates of one round (mask cm over U quads r[],
// quad u at quad index q0 + 32 u) to the list as (raw bits << 32 | ~j):
// slots from one warp scan and one shared-memory atomic per round.
template <int U>
__device__ __forceinline__ void append_round(CCtrl &ctrl, const Slice &s, const uint4 (&r)[U], uint32_t cm, int q0,
                                             uint64_t *win, uint32_t wcap, bool &over)
{
    const int lane = threadIdx.x & 31;
    const uint32_t cnt = (uint32_t)__popc(cm);
    const uint32_t ci = warp_incl_scan(cnt);
    uint32_t base = 0;
    if (lane == 31) base = atomicAdd(&ctrl.win_local, ci);
    uint32_t slot = __shfl_sync(kFull, base, 31) + ci - cnt;
    while (cm) {
        const int b = __ffs(cm) - 1;
        cm &= cm - 1u;
        const int u = b >> 2, i = b & 3;
        uint4 x = r[0];
#pragma unroll
        for (int v = 1; v < U; ++v)
            if (u == v) x = r[v];
        const uint32_t val = i == 0 ? x.x : i == 1 ? x.y : i == 2 ? x.z : x.w;
        const uint32_t j = (uint32_t)(s.jbase + 4 * (q0 + 32 * u) + i);
        if (slot < wcap) win[slot] = ((uint64_t)val << 32) | (uint64_t)(~j);
        else over = true;
        ++slot;
    }
}

// Candidate mask of a lane's round: bit 4u + i for element i of quad u.
template <int U>
__device__ __forceinline__ uint32_t cand_mask(const uint4 (&r)[U], int32_t lo_raw)
{
    uint32_t cm = 0;
#pragma unroll
    for (int u = 0; u < U; ++u)
        cm |= ((uint32_t)((int32_t)r[u].x >= lo_raw) | (uint32_t)((int32_t)r[u].y >= lo_raw) << 1 |
               (uint32_t)((int32_t)r[u].z >= lo_raw) << 2 | (uint32_t)((int32_t)r[u].w >= lo_raw) << 3)
              << (4 * u);
    return cm;
}

__device__ __forceinline__ uint32_t zero_count(const uint4 &r)
{
    return (uint32_t)(r.x == 0u) + (uint32_t)(r.y == 0u) + (uint32_t)(r.z == 0u) + (uint32_t)(r.w == 0u);
}

// The pass over the slice: keys >= lo go to the candidate list, as raw bits
// and index (finish_candidates turns them into composites and counts them
// into the fine histogram); a slot past wcap sets ctrl.overflow.  With
// PLATEAU the +0.0 entries are counted per warp in index order
// (ctrl.warp_zeros) and in all (ctrl.zeros).  lo is above the +0.0 key, so
// key >= lo holds exactly when the raw bits, read as a signed integer, are
// >= lo_raw = lo - 0x80000000 (every negative pattern is below every
// non-negative one): the scan compares raw bits, four quads per lane per
// round, and a round with no candidate in the warp costs a few instructions
// per quad.
template <int THREADS, bool PLATEAU>
__device__ void sampled_pass(CCtrl &ctrl, const Slice &s, const uint32_t *raw, const Parts &pt, uint64_t *win,
                             uint32_t wcap, uint32_t lo, int q_copy_end)
{
    constexpr int U = 4;
    constexpr int kChunkQuads = 2048;   // quads per 32 KB copy
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t lo_raw = (int32_t)(lo - 0x80000000u);
    // The copies under this warp's run of bulk-copied quads.
    {
        const int c_end = pt.q1 < q_copy_end ? pt.q1 : q_copy_end;
        if (c_end > pt.q0)
            for (int c = (pt.q0 - s.bq0) / kChunkQuads; c <= (c_end - 1 - s.bq0) / kChunkQuads; ++c)
                mbar_wait_bounded(&ctrl.bar[c], 0);
    }
    uint32_t zeros = 0;
    bool over = false;
    auto partial = [&](int q) {
        const uint32_t m = quad_mask(s, q);
        uint32_t u4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            u4[i] = !((m >> i) & 1u) ? 0xFFFFFFFFu : q < s.sq ? raw[4 * q + i] : __float_as_uint(__ldg(s.gptr + 4 * q + i));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (!((m >> i) & 1u)) continue;
            if (PLATEAU) zeros += u4[i] == 0u;
            if ((int32_t)u4[i] >= lo_raw) {
                const uint32_t slot = atomicAdd(&ctrl.win_local, 1u);
                const uint32_t j = (uint32_t)(s.jbase + 4 * q + i);
                if (slot < wcap) win[slot] = ((uint64_t)u4[i] << 32) | (uint64_t)(~j);
                else over = true;
            }
        }
    };
    if (lane == 0 && pt.head >= 0) partial(pt.head);
    // Staged quads: full rounds of U quads per lane from shared memory.
    const int q_st = pt.q1 < s.sq ? pt.q1 : (pt.q0 > s.sq ? pt.q0 : s.sq);   // end of the staged run
    const uint4 *raw4 = reinterpret_cast<const uint4 *>(raw) + lane;
    int qb = pt.q0;
    for (; qb + 32 * U <= q_st; qb += 32 * U) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r[u] = raw4[qb + 32 * u];
        int32_t mq[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            mq[u] = max(max((int32_t)r[u].x, (int32_t)r[u].y), max((int32_t)r[u].z, (int32_t)r[u].w));
        const int32_t m = max(max(mq[0], mq[1]), max(mq[2], mq[3]));
        if (PLATEAU) {
#pragma unroll
            for (int u = 0; u < U; ++u) zeros += zero_count(r[u]);
        }
        if (__any_sync(kFull, m >= lo_raw)) append_round<U>(ctrl, s, r, cand_mask<U>(r, lo_raw), qb + lane, win, wcap, over);
    }
    // The rest of the run (a partial round, and quads beyond the staging
    // area, read where they lie), with per-quad checks.
    for (; qb < pt.q1; qb += 32 * U) {
        uint4 r[U];
        uint32_t okm = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = qb + 32 * u + lane;
            r[u] = make_uint4(kFull, kFull, kFull, kFull);
            if (q < pt.q1) {
                okm |= 1u << u;
                r[u] = raw_body_quad(s, reinterpret_cast<const uint4 *>(raw), q);
            }
        }
        if (PLATEAU) {
#pragma unroll
            for (int u = 0; u < U; ++u)
                if ((okm >> u) & 1u) zeros += zero_count(r[u]);
        }
        const uint32_t cm = cand_mask<U>(r, lo_raw);   // -1 fill is below every bound
        if (__any_sync(kFull, cm != 0)) append_round<U>(ctrl, s, r, cm, qb + lane, win, wcap, over);
    }
    if (lane == 0 && pt.tail >= 0) partial(pt.tail);
    if (over) atomicOr(&ctrl.overflow, 1u);
    if (PLATEAU) {
        zeros = __reduce_add_sync(kFull, zeros);
        if (lane == 0) {
            ctrl.warp_zeros[warp] = zeros;
            if (zeros) atomicAdd(&ctrl.zeros, zeros);
        }
    }
}

// The pass in two phases, for slices of at most kMaskRounds rounds of four
// quads per lane: first each lane keeps, per round (16 entries), a 16-bit
// mask of its candidates in a register (no votes, scans or atomics in the
// scan); then one block scan of the per-thread candidate counts gives every
// thread its slots, and each thread writes its own candidates as composites
// (order key << 32 | ~j), counting each into the fine histogram.  The
// partial head and tail quads are appended first (slots by atomics).
// Counts +0.0 like sampled_pass; leaves the list length in ctrl.win_local.
constexpr int kMaskRounds = 4;

template <int THREADS>
__device__ __forceinline__ int mask_rounds(const Slice &s)
{
    constexpr int NW = THREADS / 32;
    const int n = s.bq1 - s.bq0, per = (n + NW - 1) / NW;
    return (per + 127) / 128;
}

template <int THREADS, bool PLATEAU, bool STAGED>
__device__ void masked_pass(CCtrl &ctrl, const Slice &s, const uint32_t *raw, const Parts &pt, uint64_t *win,
                            uint32_t wcap, int R, uint32_t lo, uint32_t *fhist, uint32_t f_lo, uint32_t sh,
                            int q_copy_end)
{
    constexpr int U = 4;
    constexpr int kChunkQuads = 2048;   // quads per 32 KB copy
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t lo_raw = (int32_t)(lo - 0x80000000u);
    const uint4 *raw4 = reinterpret_cast<const uint4 *>(raw);
    {
        const int c_end = pt.q1 < q_copy_end ? pt.q1 : q_copy_end;
        if (c_end > pt.q0)
            for (int c = (pt.q0 - s.bq0) / kChunkQuads; c <= (c_end - 1 - s.bq0) / kChunkQuads; ++c)
                mbar_wait_bounded(&ctrl.bar[c], 0);
    }
    uint32_t zeros = 0;
    bool over = false;
    auto put = [&](uint32_t u, uint32_t j, uint32_t slot) {
        const uint32_t e = order_key(u);
        hist_inc(fhist, fine_bin(e, f_lo, sh));
        if (slot < wcap) win[slot] = ((uint64_t)e << 32) | (uint64_t)(~j);
        else over = true;
    };
    auto partial = [&](int q) {
        const uint32_t m = quad_mask(s, q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (!((m >> i) & 1u)) continue;
            const uint32_t u = q < s.sq ? raw[4 * q + i] : __float_as_uint(__ldg(s.gptr + 4 * q + i));
            if (PLATEAU) zeros += u == 0u;
            if ((int32_t)u >= lo_raw) put(u, (uint32_t)(s.jbase + 4 * q + i), atomicAdd(&ctrl.win_local, 1u));
        }
    };
    if (lane == 0 && pt.head >= 0) partial(pt.head);
    if (lane == 0 && pt.tail >= 0) partial(pt.tail);
    // Phase 1: round r covers quads pt.q0 + 128 r + 32 u + lane.
    uint32_t mk[kMaskRounds];
    uint32_t cnt = 0;
#pragma unroll
    for (int r = 0; r < kMaskRounds; ++r) {
        mk[r] = 0u;
        if (r >= R) continue;
        const int qb = pt.q0 + 128 * r + lane;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = qb + 32 * u;
            if (q < pt.q1) {
                const uint4 x = STAGED ? raw4[q] : raw_body_quad(s, raw4, q);
                if (PLATEAU) zeros += zero_count(x);
                mk[r] |= ((uint32_t)((int32_t)x.x >= lo_raw) | (uint32_t)((int32_t)x.y >= lo_raw) << 1 |
                          (uint32_t)((int32_t)x.z >= lo_raw) << 2 | (uint32_t)((int32_t)x.w >= lo_raw) << 3)
                         << (4 * u);
            }
        }
        cnt += (uint32_t)__popc(mk[r]);
    }
    if (PLATEAU) {
        zeros = __reduce_add_sync(kFull, zeros);
        if (lane == 0) {
            ctrl.warp_zeros[warp] = zeros;
            if (zeros) atomicAdd(&ctrl.zeros, zeros);
        }
    }
    __syncthreads();   // the head and tail entries are counted
    // Phase 2: slots after the head and tail entries, in thread order.
    const uint32_t base = ctrl.win_local;
    uint32_t cnt_all;
    uint32_t slot = base + block_incl_scan1<THREADS>(cnt, ctrl.scan, cnt_all) - cnt;
    if (tid == THREADS - 1) ctrl.win_local = slot + cnt;   // read by the caller after a barrier
#pragma unroll
    for (int r = 0; r < kMaskRounds; ++r) {
        uint32_t m = mk[r];
        const int qb = pt.q0 + 128 * r + lane;
        while (m) {
            const int b = __ffs(m) - 1;
            m &= m - 1u;
            const int q = qb + 32 * (b >> 2), i = b & 3;
            const uint32_t u = STAGED || q < s.sq ? raw[4 * q + i] : __float_as_uint(__ldg(s.gptr + 4 * q + i));
            put(u, (uint32_t)(s.jbase + 4 * q + i), slot++);
        }
    }
    if (over) atomicOr(&ctrl.overflow, 1u);
}

// The CTA's candidates, appended as (raw bits << 32 | ~j), become composites
// (order key << 32 | ~j) and are counted into the fine histogram.
template <int THREADS>
__device__ __forceinline__ void finish_candidates(uint64_t *win, uint32_t n, uint32_t *fhist, uint32_t f_lo, uint32_t sh)
{
    for (uint32_t i = threadIdx.x; i < n; i += THREADS) {
        const uint64_t x = win[i];
        const uint32_t e = order_key((uint32_t)(x >> 32));
        win[i] = ((uint64_t)e << 32) | (x & 0xFFFFFFFFull);
        hist_inc(fhist, fine_bin(e, f_lo, sh));
    }
}

// The +0.0 entries of the slice in index order take output places
// n_gt + ordinal for ordinals below r, the ordinals counting from
// tie_base (the group's +0.0 entries before this CTA).  Walks the same
// per-warp parts as sampled_pass, whose per-warp counts give each warp its
// first ordinal.
template <int THREADS>
__device__ void write_zero_ties(CCtrl &ctrl, const Slice &s, const uint32_t *raw, const Parts &pt, uint32_t tie_base,
                                uint32_t r, uint32_t n_gt, uint32_t k_eff, int64_t idx_offset, int32_t *oi, float *ov,
                                bool excl)
{
    constexpr int NW = THREADS / 32;
    constexpr int U = kPassQuads;
    constexpr uint32_t kZ = 0x80000000u;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint4 *raw4 = reinterpret_cast<const uint4 *>(raw);
    if (warp == 0) {
        const uint32_t z = lane < NW ? ctrl.warp_zeros[lane] : 0u;
        const uint32_t zi = warp_incl_scan(z);
        if (lane < NW) ctrl.warp_ties[lane] = zi - z;
    }
    __syncthreads();
    uint32_t tbase = tie_base + ctrl.warp_ties[warp];
    if (ctrl.warp_zeros[warp] == 0 || tbase >= r) return;   // warp-uniform
    auto put_tie = [&](int32_t j, uint32_t ord) {
        if (ord < r && n_gt + ord < k_eff) put_out(oi, ov, n_gt + ord, idx_offset, j, kZ, excl);
    };
    auto partial = [&](int q) {
        uint32_t t = 0;
        if (lane == 0) {
            uint32_t m;
            const uint4 kk = raw_partial_keys(s, raw4, q, m);
            const uint32_t e[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (((m >> i) & 1u) && e[i] == kZ) put_tie(s.jbase + 4 * q + i, tbase + t++);
        }
        tbase += __shfl_sync(kFull, t, 0);
    };
    if (pt.head >= 0) partial(pt.head);
    for (int qb = pt.q0; qb < pt.q1 && tbase < r; qb += 32 * U) {
        uint4 kk[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = qb + u * 32 + lane;
            kk[u] = q < pt.q1 ? raw_body_keys(s, raw4, q) : make_uint4(0, 0, 0, 0);
        }
        uint32_t tm = 0;
#pragma unroll
        for (int u = 0; u < U; ++u)
            tm |= ((uint32_t)(kk[u].x == kZ) | (uint32_t)(kk[u].y == kZ) << 1 | (uint32_t)(kk[u].z == kZ) << 2 |
                   (uint32_t)(kk[u].w == kZ) << 3)
                  << (4 * u);
        if (!__any_sync(kFull, tm != 0)) continue;
        // Index order inside a round: quad u, then lane, then slot; counts
        // per u packed a byte each (at most 128) into one warp scan.
        uint32_t packed = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) packed |= (uint32_t)__popc((tm >> (4 * u)) & 0xFu) << (8 * u);
        const uint32_t ti = warp_incl_scan(packed);
        const uint32_t ttot = __shfl_sync(kFull, ti, 31), tex = ti - packed;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint32_t ord = tbase + ((tex >> (8 * u)) & 0xFFu);
            const int32_t j0 = s.jbase + 4 * (qb + u * 32 + lane);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if ((tm >> (4 * u + i)) & 1u) put_tie(j0 + i, ord++);
            tbase += (ttot >> (8 * u)) & 0xFFu;
        }
    }
    if (pt.tail >= 0 && tbase < r) partial(pt.tail);
}

// Remote stores into the shared memory of a cluster CTA (addresses from
// dsmem_addr).
__device__ __forceinline__ void dsmem_st(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_st64(uint32_t addr, uint64_t v)
{
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// The full radix select of a row group, out of line (it is the rare path of
// the cluster kernel and keeping it out of the common path keeps that path's
// code small): level 0 over the staged slice, then the threshold search and
// refinement levels, compaction, and the leader's gather, sort and write.
// Every CTA of the cluster calls it when any group of the cluster needs it,
// with work = false in the groups that are done, and runs the same cluster
// barriers.
template <int THREADS>
__device__ __noinline__ void full_select(const Params &p, const Slice &s, const RowGroup g, const bool work)
{
    constexpr uint32_t kZeroKey = 0x80000000u;   // order key of +0.0
    constexpr uint32_t kZeroDigit = kZeroKey >> 21;
    extern __shared__ __align__(16) unsigned char smem[];
    CCtrl &ctrl = *reinterpret_cast<CCtrl *>(smem);
    uint32_t *hist0 = reinterpret_cast<uint32_t *>(smem + sizeof(CCtrl));   // levels 0 and 2
    uint32_t *hist1 = hist0 + kBins;                                          // level 1
    uint64_t *win = reinterpret_cast<uint64_t *>(smem + p.off_win);
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + p.off_keys);
    const uint32_t wcap = (uint32_t)p.win_cap;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = cluster_rank();
    const int row = g.row;
    const uint32_t g0 = g.g0, gsize = g.gsize, grank = crank - g0;
    const bool leader = grank == 0;
    const int64_t rs = g.start;
    const int32_t L = g.len;
    const uint32_t k_eff = (uint32_t)(p.k < L ? p.k : L);
    const int64_t idx_offset = (p.offset_mode & TOPK_OFFSET_ROW_START) ? rs : 0;
    const bool excl = (p.offset_mode & TOPK_EXCLUDE_NEG_INF) != 0;
    int32_t *oi = p.out_idx + (int64_t)row * p.k;
    float *ov = p.out_val ? p.out_val + (int64_t)row * p.k : nullptr;
    const bool staged = s.sq == s.nq;
    const Parts pt = staged ? staged_parts<THREADS>(s, warp) : slice_parts<THREADS>(s, warp);
    const Parts ptm = slice_parts<THREADS>(s, warp);
    const uint32_t n_sentinel = (uint32_t)(4 * s.nq - (s.end - s.off0));
    {
        // Every copy has landed (the sampled pass waited on each); waiting
        // again returns at once and orders this thread after the copies.
        const int bq_end = s.bq1 < s.sq ? s.bq1 : s.sq;
        const uint32_t n_chunks = bq_end > s.bq0 ? (16u * (uint32_t)(bq_end - s.bq0) + 32767u) / 32768u : 0u;
        for (uint32_t c = 0; c < n_chunks; ++c) mbar_wait_bounded(&ctrl.bar[c], 0);
    }
    if (work) {
        for (int b = tid; b < 2 * kBins; b += THREADS) hist0[b] = 0u;
        if (tid == 0) {
            ctrl.zeros = 0u;
            ctrl.win_local = 0u;
            ctrl.wmin = kFull;
            ctrl.wmax = 0u;
        }
        __syncthreads();
        // level 0: keys in place, top-digit histogram, +0.0 counts
        if (staged) level0_pass<THREADS, true>(ctrl, s, keys, pt, hist0, n_sentinel);
        else level0_pass<THREADS, false>(ctrl, s, keys, pt, hist0, 0u);
        __syncthreads();
    }
    cluster_sync();   // B0: every CTA's level-0 histogram and counts are final

    enum { kRefine = 0, kRange = 1, kExact = 2 };
    int mode = kRefine;
    uint32_t r = k_eff, n_gt = 0, prefix = 0, lo_key = 0, T = 0, n_cand = 0;
    bool plateau = false;
    // Ties before this CTA in the group (plateau: +0.0 entries).
    auto ties_before = [&](const uint32_t *src) {
        if (warp == 0) {
            uint32_t part = lane < (int)grank ? dsmem_ld(dsmem_addr(src, g0 + (uint32_t)lane)) : 0u;
            part = __reduce_add_sync(kFull, part);
            if (lane == 0) ctrl.scan[0] = part;
        }
        __syncthreads();
        return ctrl.scan[0];
    };
    if (work) {
        if (warp == 0) {
            // The group's +0.0 count: lane l reads the group's l-th CTA.
            const uint32_t rk = g0 + (uint32_t)lane;
            uint32_t z = 0;
            if (lane < (int)gsize) z = rk == crank ? ctrl.zeros : dsmem_ld(dsmem_addr(&ctrl.zeros, rk));
            z = __reduce_add_sync(kFull, z);
            if (lane == 0) ctrl.tot[0] = z;
        }
        uint32_t d, gt, c;
        group_select<THREADS>(ctrl, hist0, g0, gsize, crank, r, d, gt, c);
        if (d == kZeroDigit && c == ctrl.tot[0]) {
            // The boundary bin holds only +0.0: the k-th key is +0.0.
            mode = kExact;
            plateau = true;
            T = kZeroKey;
            n_gt = gt;
            r -= gt;
        } else if (gt + c <= wcap) {
            mode = kRange;
            lo_key = d << 21;
            n_cand = gt + c;
        } else {
            prefix = d;
            n_gt = gt;
            r -= gt;
        }
        if (mode != kRefine) {
            if (plateau)
                compact<THREADS, true>(staged, ctrl, s, keys, pt, ptm, win, wcap, 0u, T, ties_before(&ctrl.zeros), r,
                                       n_gt, k_eff, idx_offset, oi, ov, excl);
            else
                compact<THREADS, false>(staged, ctrl, s, keys, pt, ptm, win, wcap, lo_key, 0u, 0u, r, n_gt, k_eff,
                                        idx_offset, oi, ov, excl);
        } else {
            refine_pass<THREADS>(staged, s, keys, pt, ptm, hist1, prefix, 21, 10, 0x7FFu);
            __syncthreads();
        }
    }
    cluster_sync();   // B1

    if (work && mode == kRefine) {
        uint32_t d, gt, c;
        group_select<THREADS>(ctrl, hist1, g0, gsize, crank, r, d, gt, c);
        if (n_gt + gt + c <= wcap) {
            mode = kRange;
            lo_key = (prefix << 21) | (d << 10);
            n_cand = n_gt + gt + c;
            compact<THREADS, false>(staged, ctrl, s, keys, pt, ptm, win, wcap, lo_key, 0u, 0u, r, n_gt, k_eff,
                                    idx_offset, oi, ov, excl);
        } else {
            prefix = (prefix << 11) | d;
            n_gt += gt;
            r -= gt;
            // Every peer pulled hist0 before B1: it can be reused.
            for (int b = tid; b < kBins; b += THREADS) hist0[b] = 0u;
            __syncthreads();
            refine_pass<THREADS>(staged, s, keys, pt, ptm, hist0, prefix, 10, 0, 0x3FFu);
            __syncthreads();
        }
    }
    cluster_sync();   // B2

    if (work && mode == kRefine) {
        uint32_t d, gt, c;
        group_select<THREADS>(ctrl, hist0, g0, gsize, crank, r, d, gt, c);
        mode = kExact;
        T = (prefix << 10) | d;
        n_gt += gt;
        r -= gt;
        const uint32_t tb = ties_before(&hist0[T & 0x3FFu]);
        compact<THREADS, true>(staged, ctrl, s, keys, pt, ptm, win, wcap, 0u, T, tb, r, n_gt, k_eff, idx_offset, oi,
                               ov, excl);
    }
    cluster_sync();   // B3: every CTA's candidate list is final

    // ---- 7. the leader gathers the group's lists into its staging area
    //         (its own keys are no longer needed), releases the peers and
    //         sorts; the peers wait until it has read their lists ---------- //
    uint64_t *cand = reinterpret_cast<uint64_t *>(keys);
    uint32_t n = 0;
    if (work && leader) {
        if (warp == 0) {
            const uint32_t rk = g0 + (uint32_t)lane;
            uint32_t cnt = 0, mn = kFull, mx = 0;
            if (lane < (int)gsize) {
                cnt = rk == crank ? ctrl.win_local : dsmem_ld(dsmem_addr(&ctrl.win_local, rk));
                mn = rk == crank ? ctrl.wmin : dsmem_ld(dsmem_addr(&ctrl.wmin, rk));
                mx = rk == crank ? ctrl.wmax : dsmem_ld(dsmem_addr(&ctrl.wmax, rk));
            }
            cnt = min(cnt, wcap);
            const uint32_t incl = warp_incl_scan(cnt);
            ctrl.warp_ties[lane] = incl - cnt;   // offset of the group's CTA `lane`
            ctrl.warp_zeros[lane] = cnt;
            mn = __reduce_min_sync(kFull, mn);
            mx = __reduce_max_sync(kFull, mx);
            if (lane == 31) ctrl.sel[0] = incl;
            if (lane == 0) {
                ctrl.sel[1] = mn;
                ctrl.sel[2] = mx;
            }
        }
        __syncthreads();
        n = ctrl.sel[0];
        for (uint32_t gr = 0; gr < gsize; ++gr) {
            const uint32_t cnt = ctrl.warp_zeros[gr], off = ctrl.warp_ties[gr];
            if (off + cnt > wcap) continue;   // flagged below
            if (gr == 0) {
                for (uint32_t i = tid; i < cnt; i += THREADS) cand[off + i] = win[i];
            } else {
                const uint32_t src = dsmem_addr(win, g0 + gr);
                for (uint32_t i = tid; i < cnt; i += THREADS) cand[off + i] = dsmem_ld64(src + 8u * i);
            }
        }
        __syncthreads();
    }
    cluster_arrive();   // B4: the leaders have read every list
    if (work && leader) {
        const uint32_t expect = mode == kRange ? n_cand : n_gt;
        if (n != expect || n > wcap) {
            if (tid == 0) atomicOr(&g_status, TOPK_DEV_INTERNAL);
            n = min(min(n, expect), wcap);
        }
        const uint32_t n_o = mode == kRange ? k_eff : n_gt;
        if (n > 0) {
            sort_and_write<THREADS>(cand, win, (int)n, (int)min(n, n_o), (int)wcap, ctrl.sel[1], ctrl.sel[2], hist0,
                                    ctrl.scan64, oi, ov, idx_offset, excl);
        }
        pad_out(oi, ov, (int)k_eff, p.k);
        if (p.page_table) {   // the peers' tie writes are visible since B3
            __syncthreads();
            page_map_row(p, row, oi, (int)k_eff);
        }
    }
    cluster_wait();
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS, 2048 / THREADS / 2) topk_cluster_kernel(const Params p)
{
    grid_dependency_enter();
    constexpr uint32_t kZeroKey = 0x80000000u;   // order key of +0.0
    constexpr uint32_t kChunk = 32768;           // bytes per bulk copy
    extern __shared__ __align__(16) unsigned char smem[];
    CCtrl &ctrl = *reinterpret_cast<CCtrl *>(smem);
    uint32_t *hist0 = reinterpret_cast<uint32_t *>(smem + sizeof(CCtrl));   // levels 0 and 2
    uint64_t *win = reinterpret_cast<uint64_t *>(smem + p.off_win);
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + p.off_keys);
    const uint32_t wcap = (uint32_t)p.win_cap;   // candidate list capacity (a power of two)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = cluster_rank(), csize = cluster_size();
    // The row plan's scratch is the candidate list, which only this CTA
    // writes (peers push into the histograms before the first cluster
    // barrier, and into the staging area after it).
    const RowGroup g = assign_rows<THREADS>(p, crank, csize, reinterpret_cast<uint32_t *>(win), ctrl.scan);
    if (g.row < 0) return;   // uniform over the cluster: nothing to select
    const int row = g.row;
    const uint32_t g0 = g.g0, gsize = g.gsize, grank = crank - g0;
    const bool leader = grank == 0;

    // Rows handed out by assign_rows have 0 < L < 2^24 and a valid window.
    const int64_t rs = g.start;
    const int32_t L = g.len;
    const uint32_t k_eff = (uint32_t)(p.k < L ? p.k : L);
    const int64_t idx_offset = (p.offset_mode & TOPK_OFFSET_ROW_START) ? rs : 0;
    const bool excl = (p.offset_mode & TOPK_EXCLUDE_NEG_INF) != 0;
    int32_t *oi = p.out_idx + (int64_t)row * p.k;
    float *ov = p.out_val ? p.out_val + (int64_t)row * p.k : nullptr;

    Slice s;
    {
        const uint64_t pa = (uint64_t)(uintptr_t)p.scores >> 2;   // element address
        const int64_t e0 = rs, e1 = rs + L;
        int64_t a0 = e0 + (int64_t)((4u - (uint32_t)((pa + (uint64_t)e0) & 3u)) & 3u);
        if (a0 > e1) a0 = e1;
        const int64_t n4 = (e1 - a0) >> 2;
        // n4 < 2^22 and gsize <= 16: the products fit 32 bits.
        const int64_t qlo = (uint32_t)n4 * grank / gsize, qhi = (uint32_t)n4 * (grank + 1) / gsize;
        const int64_t hb = a0 + 4 * qlo, he = a0 + 4 * qhi;
        const int64_t glo = grank == 0 ? e0 : hb;
        const int64_t ghi = grank == gsize - 1 ? e1 : he;
        const int64_t sbase = hb - ((hb - glo + 3) & ~(int64_t)3);
        s.gptr = p.scores + sbase;
        s.off0 = (int32_t)(glo - sbase);
        s.end = (int32_t)(ghi - sbase);
        s.bq0 = (int32_t)((hb - sbase) >> 2);
        s.bq1 = (int32_t)((he - sbase) >> 2);
        s.nq = (s.end + 3) >> 2;
        s.sq = s.nq < (p.stage_cap >> 2) ? s.nq : (p.stage_cap >> 2);
        s.jbase = (int32_t)(sbase - rs);
    }
    // Each warp's contiguous run of the slice's full quads, with the
    // partial head quad in warp 0 and the partial tail quad in the last.
    const Parts ptm = slice_parts<THREADS>(s, warp);

    // ---- 1. the row's sample, then the bulk copies (TMA) of the staged
    //         body; the sample and the partial head and tail quads are
    //         read with plain loads into registers, the sample first so
    //         that it is not queued behind the copies ------------------- //
    // The sample: the whole row when L <= kSample, else 128 runs of 32
    // consecutive scores spread evenly over the row (run t starts at
    // t * (L - 32) / 127), so that it costs a few cache lines per row rather
    // than a read of most of the row's DRAM bursts.  The same in every CTA
    // of the group (raw bits; keys after the barrier).
    constexpr int SPT = kSample / THREADS;
    static_assert(kPassQuads == 2, "the append step reads the round's two quads");
    const uint32_t S = (uint32_t)(L < kSample ? L : kSample);
    uint32_t skey[SPT];
#pragma unroll
    for (int u = 0; u < SPT; ++u) {
        const uint32_t t = (uint32_t)tid + (uint32_t)(u * THREADS);
        const uint32_t j = L <= kSample ? t : (t >> 5) * (uint32_t)(L - 32) / 127u + (t & 31u);
        skey[u] = t < S ? __float_as_uint(__ldg(p.scores + rs + j)) : 0u;
    }
    // One mbarrier per 32 KB copy, so that each warp can start on its part
    // of the slice as soon as the copies under it have landed.
    const int bq_end = s.bq1 < s.sq ? s.bq1 : s.sq;
    const uint32_t copy_bytes = bq_end > s.bq0 ? 16u * (uint32_t)(bq_end - s.bq0) : 0u;
    const uint32_t n_chunks = (copy_bytes + kChunk - 1) / kChunk;   // at most 8 (shared memory < 256 KB)
    // Lane 0 of warp c issues chunk c, so the copies start side by side.
    if (lane == 0 && (uint32_t)warp < n_chunks) {
        const uint32_t c = (uint32_t)warp;
        const uint32_t off = c * kChunk, len = copy_bytes - off < kChunk ? copy_bytes - off : kChunk;
        mbar_init(&ctrl.bar[c], 1);
        mbar_init_fence();
        mbar_arrive_expect_tx(&ctrl.bar[c], len);
        bulk_load(reinterpret_cast<unsigned char *>(keys + 4 * s.bq0) + off,
                  reinterpret_cast<const unsigned char *>(s.gptr + 4 * s.bq0) + off, len, &ctrl.bar[c]);
    }
    // Staged quads outside the body: at most one head and one tail quad,
    // raw bits with 0xFFFFFFFF (order key 0) in the empty slots.
    const int pq_q = tid < 1 ? 0 : s.nq - 1;
    const bool pq_mine = tid < 2 && pq_q < s.sq && (pq_q < s.bq0 || pq_q >= s.bq1);
    uint32_t pq[4] = {kFull, kFull, kFull, kFull};
    if (pq_mine) {
        const uint32_t m = quad_mask(s, pq_q);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if ((m >> i) & 1u) pq[i] = __float_as_uint(__ldg(s.gptr + 4 * pq_q + i));
    }
    // Fine histograms: hist0 and hist1 hold four slots of kFineBins words.
    // A group of up to four CTAs keeps all of its CTAs' histograms in every
    // CTA: each counts into its own slot (grank) and writes that slot into
    // its peers before the cluster barrier.  A larger group counts into
    // slot 3, which its peers read after the barrier.  Nothing but a CTA's
    // own counting slot is touched before the barrier, so the peers' writes
    // cannot race with it.  The sample's histograms use the candidate-list
    // area, which holds no candidates yet.
    const bool push_mode = gsize <= 4;
    uint32_t *fine = hist0;                                    // 4 slots of kFineBins
    uint32_t *fhist = fine + (push_mode ? grank : 3u) * kFineBins;
    uint32_t *sh0 = reinterpret_cast<uint32_t *>(win);   // 4096 bins (the list holds at least 2048 composites)
    for (int b = tid; b < kFineBins; b += THREADS) fhist[b] = 0u;
    for (int b = tid; b < 4096; b += THREADS) sh0[b] = 0u;
    if (tid == 0) {
        ctrl.zeros = 0u;
        ctrl.win_local = 0u;
        ctrl.smax = 0u;
        ctrl.overflow = 0u;
        ctrl.cl_fb = 0u;
        ctrl.maxbin = 0u;
        ctrl.loc_begin = kFull;
        ctrl.loc_end = 0u;
        ctrl.smin = kFull;
    }
    __syncthreads();

    // ---- 2. the candidate bound: the top 12 bits (an eighth of a binade)
    //         of the sample's m-th largest key (m = k when the sample is the
    //         whole row), from a 4096-bin histogram of the sample ----------- //
    constexpr int kSampleBins = 4096;
    {
        uint32_t smx = 0, smn = kFull;
#pragma unroll
        for (int u = 0; u < SPT; ++u) {
            if ((uint32_t)tid + (uint32_t)(u * THREADS) < S) {
                skey[u] = order_key(skey[u]);
                hist_inc(sh0, skey[u] >> 20);
                smx = max(smx, skey[u]);
                if (skey[u] > kZeroKey) smn = min(smn, skey[u]);
            }
        }
        smx = __reduce_max_sync(kFull, smx);
        smn = __reduce_min_sync(kFull, smn);
        // smin takes the smallest sampled positive key; a part-row
        // sample's lies above the row's, so the plateau path's fine range
        // starts four binades lower (not below the smallest positive key).
        if (L > kSample && smn != kFull) smn -= min(smn - (kZeroKey + 1u), 4u << 23);
        if (lane == 0) {
            atomicMax(&ctrl.smax, smx);
            atomicMin(&ctrl.smin, smn);
        }
    }
    __syncthreads();
    uint32_t m_s = k_eff;
    if (L > kSample) {
        const float q = (float)k_eff / (float)L;
        const float mu = (float)S * q;
        const float m = ceilf(mu + 4.0f * sqrtf(mu * (1.0f - q)) + 8.0f);
        m_s = m < (float)S ? (uint32_t)m : S;
    }
    {
        uint32_t d, gt;
        if (find_bin_nb<THREADS, kSampleBins>(sh0, m_s, ctrl.scan, d, gt)) ctrl.sel[0] = d;
    }
    __syncthreads();
    // A bound on or below the +0.0 digit makes the candidates the positive
    // keys, with +0.0 counted apart.  Candidates are the keys >= lo; fine
    // bins start at f_lo (on the plateau path the smallest sampled positive
    // key, lowered as above).
    const uint32_t d1 = ctrl.sel[0];
    const bool plat = d1 <= (kZeroKey >> 20);
    const uint32_t lo = plat ? kZeroKey + 1u : d1 << 20;
    const uint32_t f_lo = plat ? (ctrl.smin != kFull ? ctrl.smin : lo) : lo;
    const uint32_t smax = ctrl.smax;
    // The sample's range spans 1024 fine bins when few keys can lie above
    // its largest (about L / S of them), else 512, which leaves the upper
    // half of the bins to those keys.
    const int span_bits = 32 - __clz(smax > f_lo ? smax - f_lo : 0u);
    const int fine_bits = L > 64 * kSample ? 9 : 10;
    const uint32_t sh = span_bits > fine_bits ? (uint32_t)(span_bits - fine_bits) : 0u;
    if (pq_mine) {
#pragma unroll
        for (int i = 0; i < 4; ++i) keys[4 * pq_q + i] = pq[i];
    }
    __syncthreads();   // the partial quads are staged; every thread has read ctrl.smin and ctrl.sel

    // ---- 3. one pass: candidates to the fine histogram and the list ------ //
    // Slices of up to kMaskRounds rounds per lane take the two-phase pass,
    // which also writes the composites and the fine histogram; longer ones
    // the appending pass, finished below.
    const int mask_r = mask_rounds<THREADS>(s);
    const uint32_t wcap_eff = wcap;
    if (mask_r <= kMaskRounds) {
        if (s.sq == s.nq) {
            if (plat) masked_pass<THREADS, true, true>(ctrl, s, keys, ptm, win, wcap, mask_r, lo, fhist, f_lo, sh, bq_end);
            else masked_pass<THREADS, false, true>(ctrl, s, keys, ptm, win, wcap, mask_r, lo, fhist, f_lo, sh, bq_end);
        } else {
            if (plat) masked_pass<THREADS, true, false>(ctrl, s, keys, ptm, win, wcap, mask_r, lo, fhist, f_lo, sh, bq_end);
            else masked_pass<THREADS, false, false>(ctrl, s, keys, ptm, win, wcap, mask_r, lo, fhist, f_lo, sh, bq_end);
        }
        __syncthreads();
    } else {
        if (plat) sampled_pass<THREADS, true>(ctrl, s, keys, ptm, win, wcap, lo, bq_end);
        else sampled_pass<THREADS, false>(ctrl, s, keys, ptm, win, wcap, lo, bq_end);
        __syncthreads();
        finish_candidates<THREADS>(win, min(ctrl.win_local, wcap), fhist, f_lo, sh);
        __syncthreads();
    }

    // ---- 4. counters (and, for small groups, the fine histogram) into
    //         every CTA of the group ---------------------------------------- //
    if (tid < (int)gsize) {
        const uint32_t dst = g0 + (uint32_t)tid;
        const uint32_t v[3] = {ctrl.win_local, ctrl.overflow, ctrl.zeros};
        uint32_t *fld[3] = {&ctrl.gcnt[grank], &ctrl.gover[grank], &ctrl.gzero[grank]};
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            if (dst == crank) *fld[i] = v[i];
            else dsmem_st(dsmem_addr(fld[i], dst), v[i]);
        }
    }
    if (push_mode) {
        for (uint32_t r0 = g0; r0 < g0 + gsize; ++r0) {
            if (r0 == crank) continue;
            for (int b = tid; b < kFineBins; b += THREADS) dsmem_st(dsmem_addr(&fhist[b], r0), fhist[b]);
        }
    }
    cluster_sync();   // F0: every CTA's list, counters and fine histogram are in place

    // ---- 5. the group's totals, every fine bin's first output place ------ //
    uint32_t n_all = 0, z_all = 0, z_before = 0, over_any = 0;
    for (uint32_t gr = 0; gr < gsize; ++gr) {
        n_all += ctrl.gcnt[gr];
        z_all += ctrl.gzero[gr];
        z_before += gr < grank ? ctrl.gzero[gr] : 0u;
        over_any |= ctrl.gover[gr];
    }
    // The output places the sampled path fills: all k_eff, or on the
    // plateau path with fewer positives than k_eff the positives (the first
    // +0.0 entries follow them).
    uint32_t n_out = k_eff, r_ties = 0;
    bool fast = over_any == 0u;
    if (n_all < k_eff) {
        if (plat && n_all + z_all >= k_eff) {
            n_out = n_all;
            r_ties = k_eff - n_all;
        } else {
            fast = false;
        }
    }
    const uint32_t pos_lo = n_out * grank / gsize;   // n_out <= 4096, gsize <= 16: products fit 32 bits
    const uint32_t pos_hi = n_out * (grank + 1) / gsize;
    if (tid <= (int)gsize) ctrl.gpos[tid] = n_out * (uint32_t)tid / gsize;
    constexpr int FB = kFineBins / THREADS;
    const int flo = kFineBins - (tid + 1) * FB;   // thread 0 owns the top bins
    uint32_t *offs = fine;                        // slot 0: first output place of each bin
    uint32_t *base = fine + kFineBins;            // slot 1: the bin's members in lower CTAs
    uint32_t *lcur = fine + 2 * kFineBins;        // slot 2: this CTA's members placed so far
    uint32_t n_bins_total;                        // candidates counted in the group's fine bins
    {
        uint32_t h[FB], hb[FB];
#pragma unroll
        for (int i = 0; i < FB; ++i) {
            h[i] = 0u;
            hb[i] = 0u;
        }
        for (uint32_t gr = 0; gr < gsize; ++gr) {
#pragma unroll
            for (int i = 0; i < FB; ++i) {
                uint32_t v;
                if (push_mode) v = fine[gr * kFineBins + flo + i];
                else v = g0 + gr == crank ? fhist[flo + i] : dsmem_ld(dsmem_addr(&fhist[flo + i], g0 + gr));
                h[i] += v;
                hb[i] += gr < grank ? v : 0u;
            }
        }
        uint32_t hs = 0, hmax = 0;
#pragma unroll
        for (int i = 0; i < FB; ++i) {
            hs += h[i];
            hmax = max(hmax, h[i]);
        }
        hmax = __reduce_max_sync(kFull, hmax);
        if (lane == 0) atomicMax(&ctrl.maxbin, hmax);
        uint32_t run = block_incl_scan1<THREADS>(hs, ctrl.scan, n_bins_total) - hs;
        // Every thread rewrites only its own bins of slots 0-2, whose
        // pushed counts it has read above.
        uint32_t lb = kFull, le = 0;
#pragma unroll
        for (int i = FB - 1; i >= 0; --i) {
            offs[flo + i] = run;
            base[flo + i] = hb[i];
            lcur[flo + i] = 0u;
            if (h[i] > 0 && run >= pos_lo && run < pos_hi && run < n_out) {
                lb = min(lb, run - pos_lo);
                le = max(le, run + h[i] - pos_lo);
            }
            run += h[i];
        }
        lb = __reduce_min_sync(kFull, lb);
        le = __reduce_max_sync(kFull, le);
        if (lane == 0 && le > 0) {
            atomicMin(&ctrl.loc_begin, lb);
            atomicMax(&ctrl.loc_end, le);
        }
    }
    __syncthreads();
    // With no list overflow every candidate was counted once (an overflow
    // leaves the rest uncounted and sends the group to the full select).
    if (over_any == 0u && n_all != n_bins_total && tid == 0) atomicOr(&g_status, TOPK_DEV_INTERNAL);
    const uint32_t loc_cap = (uint32_t)p.stage_cap / 2u;   // composites the staging area holds
    fast = fast && n_all == n_bins_total && n_all <= loc_cap && ctrl.maxbin <= kMaxFineBin;

    // ---- 6. sampled path: every candidate to the CTA owning its bin's
    //         first place, at its bin's place range ------------------------ //
    uint64_t *loc = reinterpret_cast<uint64_t *>(keys);   // the staged slice becomes the gather buffer
    // A row of one CTA places its first +0.0 entries now, from the staged
    // slice (no peer writes into this CTA); a larger group does it after F1
    // from the scores where they lie, since its peers' candidates land in the
    // staging area.
    const bool ties_now = fast && r_ties > 0 && gsize == 1;
    if (ties_now) {
        write_zero_ties<THREADS>(ctrl, s, keys, ptm, z_before, r_ties, n_out, k_eff, idx_offset, oi, ov, excl);
        __syncthreads();   // the slice has been read
    }
    if (fast) {
        const uint32_t cnt = min(ctrl.win_local, wcap_eff);
        for (uint32_t i = (uint32_t)tid; i < cnt; i += THREADS) {
            const uint64_t c = win[i];
            const uint32_t f = fine_bin((uint32_t)(c >> 32), f_lo, sh);
            const uint32_t o = offs[f];
            if (o >= n_out) continue;   // the bin starts past the output
            uint32_t gr = 0;
            while (gr + 1 < gsize && ctrl.gpos[gr + 1] <= o) ++gr;
            const uint32_t slot = o + base[f] + atomicAdd(&lcur[f], 1u);
            const uint32_t dst = slot - ctrl.gpos[gr];
            if (gr == grank) loc[dst] = c;
            else dsmem_st64(dsmem_addr(&loc[dst], g0 + gr), c);
        }
    } else if (tid < (int)csize) {
        dsmem_st(dsmem_addr(&ctrl.cl_fb, (uint32_t)tid), 1u);   // the cluster runs the full select below
    }
    cluster_sync();   // F1: every candidate is with its bin's CTA; every fallback flag is set
    const bool cluster_fallback = ctrl.cl_fb != 0u;
    if (fast) {
        // A bin's members sit together at [offs, offs + count) - pos_lo; a
        // member's place is the bin's first place plus the members above it.
        const uint32_t loc_end = ctrl.loc_end;
        for (uint32_t i = ctrl.loc_begin + (uint32_t)tid; i < loc_end; i += THREADS) {
            const uint64_t x = loc[i];
            const uint32_t e = (uint32_t)(x >> 32);
            const uint32_t f = fine_bin(e, f_lo, sh);
            const uint32_t st = offs[f] - pos_lo, en = (f > 0 ? offs[f - 1] : n_all) - pos_lo;
            uint32_t rank = 0;
            for (uint32_t y = st; y < en; ++y) rank += loc[y] > x;
            const uint32_t pos = offs[f] + rank;
            if (pos < n_out) put_out(oi, ov, pos, idx_offset, (int32_t)(~(uint32_t)x), e, excl);
        }
        if (r_ties > 0 && !ties_now) {
            // The first +0.0 entries by index, read where they lie (the
            // staging area now holds the gathered candidates).
            Slice sg = s;
            sg.sq = 0;
            write_zero_ties<THREADS>(ctrl, sg, keys, ptm, z_before, r_ties, n_out, k_eff, idx_offset, oi, ov, excl);
        }
        if (leader) pad_out(oi, ov, (int)k_eff, p.k);
    }
    if (p.page_table) {
        __syncthreads();
        cluster_sync();   // the group's output writes are done
        if (fast && leader) page_map_row(p, row, oi, (int)k_eff);
    }
    if (!cluster_fallback) return;

    // ---- 7. the full radix select, for the groups whose checks failed;
    //         every CTA of the cluster runs the same cluster barriers ------ //
    full_select<THREADS>(p, s, g, !fast);
}

// ------------------------------------------------------------------------- //
// Tie / plateau statistics of each row at its k-th boundary, one cluster of
// CS CTAs per row (CS = 1..16, from B on the host).  The radix select of the
// top-k kernels, every pass reading the row from global memory: each CTA
// bins its contiguous slice, the cluster's histograms are summed over DSMEM
// after a cluster barrier, and every CTA makes the same selection from the
// same integers.  The top 11, next 11 and last 10 bits of the order key
// narrow the bin holding the k-th key down to the key itself; the entries
// above it and equal to it are the counts above and inside the last bin.
// Levels 0 and 2 use one histogram buffer and level 1 the other, so one
// cluster barrier per level keeps every CTA's reads ahead of the next
// clear.  A row no longer than k takes one pass (its 0.0 count).
// ------------------------------------------------------------------------- //
constexpr int kStatsThreads = 512;

template <int THREADS>
__global__ void __launch_bounds__(THREADS) topk_stats_cluster_kernel(const float *scores, int64_t n_scores,
                                                                     const int32_t *row_starts,
                                                                     const int32_t *lengths, int32_t k,
                                                                     topk_row_stats *out)
{
    grid_dependency_enter();
    constexpr int BPT = kBins / THREADS;
    static_assert(BPT == 4, "four bins per thread: one 16-byte DSMEM load per peer");
    constexpr uint32_t kNone = 0xFFFFFFFFu;
    __shared__ __align__(16) uint32_t hist[2][kBins];
    __shared__ uint32_t scan[32];
    __shared__ uint32_t sel[3];   // selected digit, entries above its bin, entries in it
    __shared__ uint32_t zeros;    // this CTA's 0.0 count
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t crank = cluster_rank(), csize = cluster_size();
    const int row = (int)(blockIdx.x / csize);

    topk_row_stats res = {0u, 0u, 0u, 0u, 0u, 0u};
    const int64_t rs = row_starts[row];
    int64_t len = lengths[row];
    if (len < 0) len = 0;
    uint32_t bad = 0;
    if (len >= (int64_t)TOPK_RAGGED_MAX_LEN)
        bad = TOPK_DEV_LEN_ENVELOPE;
    else if (rs < 0 || rs + len > n_scores)
        bad = TOPK_DEV_BAD_WINDOW;
    if (bad) {   // the same for every CTA of the cluster: none touches another's memory
        if (crank == 0 && tid == 0) {
            atomicOr(&g_status, bad);
            out[row] = res;
        }
        return;
    }
    const uint32_t L = (uint32_t)len;
    const bool has_boundary = L > (uint32_t)k;

    // This CTA's slice as [head | 16-byte aligned quads | tail]; head and
    // tail hold fewer than four entries each.
    const uint32_t lo = (uint32_t)((uint64_t)L * crank / csize);
    const uint32_t Ls = (uint32_t)((uint64_t)L * (crank + 1) / csize) - lo;
    const float *x = scores + rs + lo;
    const uint32_t *xs = reinterpret_cast<const uint32_t *>(x);
    const uint32_t head = min(Ls, (4u - (uint32_t)(((uintptr_t)x >> 2) & 3u)) & 3u);
    const uint32_t nq = (Ls - head) >> 2;
    const uint32_t tail0 = head + 4u * nq;
    const uint4 *xq = reinterpret_cast<const uint4 *>(x + head);

    if (tid == 0) zeros = 0u;
    uint32_t prefix = 0, above = 0, r = (uint32_t)k, tie = 0;
    bool failed = false;
    const int levels = has_boundary ? 3 : 1;
    for (int level = 0; level < levels; ++level) {
        const int dsh = level == 0 ? 21 : (level == 1 ? 10 : 0);   // digit shift
        const int dbits = level == 2 ? 10 : 11;
        const uint32_t dmask = (1u << dbits) - 1u;
        uint32_t *H = hist[level == 1 ? 1 : 0];
        for (int b = tid; b < kBins; b += THREADS) H[b] = 0u;
        if (tid == 0) {
            sel[0] = kNone;
            sel[1] = 0u;
            sel[2] = 0u;
        }
        __syncthreads();

        // Level 0 counts 0.0 entries and bins every entry; later levels bin
        // the entries whose higher bits equal the selected prefix.
        uint32_t nz = 0;
        auto visit = [&](uint32_t u) {
            const uint32_t key = order_key(u);
            if (level == 0) {
                nz += (u & 0x7FFFFFFFu) == 0u;
                if (has_boundary) atomicAdd(&H[key >> 21], 1u);
            } else if ((key >> (dsh + dbits)) == prefix) {
                atomicAdd(&H[(key >> dsh) & dmask], 1u);
            }
        };
        if ((uint32_t)tid < head) visit(xs[tid]);
        for (uint32_t q = (uint32_t)tid; q < nq; q += 4u * THREADS) {
            uint4 v[4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
                v[t] = q + t * THREADS < nq ? __ldg(xq + q + t * THREADS) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (q + t * THREADS < nq) {
                    visit(v[t].x);
                    visit(v[t].y);
                    visit(v[t].z);
                    visit(v[t].w);
                }
            }
        }
        if (tail0 + (uint32_t)tid < Ls) visit(xs[tail0 + tid]);
        if (level == 0) {
            nz = __reduce_add_sync(kFull, nz);
            if (lane == 0 && nz) atomicAdd(&zeros, nz);
        }
        cluster_sync();   // every CTA's histogram (and 0.0 count) of this level is final
        if (!has_boundary) break;

        // The cluster's bins, top first: thread t holds bins kBins-1-4t down
        // to kBins-4(t+1), summed over the cluster's CTAs in rank order.
        uint32_t h[BPT] = {0u, 0u, 0u, 0u};
        const uint32_t *hb = &H[kBins - BPT * (tid + 1)];
        for (uint32_t q = 0; q < csize; ++q) {
            uint32_t v[4];
            dsmem_ld_bins(dsmem_addr(hb, q), v);
            h[0] += v[3];
            h[1] += v[2];
            h[2] += v[1];
            h[3] += v[0];
        }
        const uint32_t sum = h[0] + h[1] + h[2] + h[3];
        uint32_t run = block_incl_scan<THREADS>(sum, scan) - sum;
#pragma unroll
        for (int i = 0; i < BPT; ++i) {
            if (run < r && run + h[i] >= r) {   // the bin where the count from the top reaches r
                sel[0] = (uint32_t)(kBins - 1 - (BPT * tid + i));
                sel[1] = run;
                sel[2] = h[i];
            }
            run += h[i];
        }
        __syncthreads();
        const uint32_t d = sel[0];
        if (d == kNone) {   // cannot happen: the selected bin always holds >= r entries
            failed = true;
            break;
        }
        above += sel[1];
        r -= sel[1];
        prefix = (prefix << dbits) | d;
        if (level == 2) tie = sel[2];
        __syncthreads();   // every thread has read sel
    }
    if (crank == 0 && tid == 0) {
        uint32_t nzero = 0;
        for (uint32_t q = 0; q < csize; ++q) nzero += dsmem_ld(dsmem_addr(&zeros, q));
        if (failed) {
            atomicOr(&g_status, TOPK_DEV_INTERNAL);
        } else {
            res.len = L;
            res.n_zero = nzero;
            if (has_boundary) {
                const uint32_t T = prefix;   // the k-th key
                res.boundary_bits = key_bits(T);
                res.tie = tie;
                res.above = above;
                res.flags = TOPK_STAT_HAS_BOUNDARY;
                if (tie > 1u && above + tie > (uint32_t)k) res.flags |= TOPK_STAT_STRADDLE;
                if ((res.boundary_bits & 0x7FFFFFFFu) == 0u) res.flags |= TOPK_STAT_ZERO_BOUND;
            } else {
                res.above = L;
            }
        }
        out[row] = res;
    }
    cluster_sync();   // no CTA leaves while a peer may still read its shared memory
}

// ------------------------------------------------------------------------- //
// The one-CTA form of the statistics kernel, for batches of many rows (or
// short ones): one CTA per row.  The radix select of the top-k kernels, with every pass reading the
// row from global memory: the top 11, next 11 and last 10 bits of the order
// key narrow the bin holding the k-th key down to the key itself, and the
// entries above it and equal to it are the counts above and inside the last
// bin.  A row no longer than k takes one pass (its 0.0 count).
// ------------------------------------------------------------------------- //
template <int THREADS>
__global__ void __launch_bounds__(THREADS) topk_stats_kernel(const float *scores, int64_t n_scores,
                                                             const int32_t *row_starts, const int32_t *lengths,
                                                             int32_t k, topk_row_stats *out)
{
    grid_dependency_enter();
    constexpr int BPT = kBins / THREADS;
    constexpr uint32_t kNone = 0xFFFFFFFFu;
    __shared__ uint32_t hist[kBins];
    __shared__ uint32_t scan[32];
    __shared__ uint32_t sel[3];   // selected digit, entries above its bin, 0.0 count
    const int tid = threadIdx.x, lane = tid & 31;
    const int row = (int)blockIdx.x;

    topk_row_stats res = {0u, 0u, 0u, 0u, 0u, 0u};
    const int64_t rs = row_starts[row];
    int64_t len = lengths[row];
    if (len < 0) len = 0;
    uint32_t bad = 0;
    if (len >= (int64_t)TOPK_RAGGED_MAX_LEN)
        bad = TOPK_DEV_LEN_ENVELOPE;
    else if (rs < 0 || rs + len > n_scores)
        bad = TOPK_DEV_BAD_WINDOW;
    if (bad) {
        if (tid == 0) {
            atomicOr(&g_status, bad);
            out[row] = res;
        }
        return;
    }
    const uint32_t L = (uint32_t)len;
    const bool has_boundary = L > (uint32_t)k;

    // The row as [head | 16-byte aligned quads | tail]; head and tail hold
    // fewer than four entries each.
    const float *x = scores + rs;
    const uint32_t *xs = reinterpret_cast<const uint32_t *>(x);
    const uint32_t head = min(L, (4u - (uint32_t)(((uintptr_t)x >> 2) & 3u)) & 3u);
    const uint32_t nq = (L - head) >> 2;
    const uint32_t tail0 = head + 4u * nq;
    const uint4 *xq = reinterpret_cast<const uint4 *>(x + head);

    uint32_t prefix = 0, above = 0, r = (uint32_t)k, tie = 0;
    const int levels = has_boundary ? 3 : 1;
    for (int level = 0; level < levels; ++level) {
        const int dsh = level == 0 ? 21 : (level == 1 ? 10 : 0);   // digit shift
        const int dbits = level == 2 ? 10 : 11;
        const uint32_t dmask = (1u << dbits) - 1u;
        for (int b = tid; b < kBins; b += THREADS) hist[b] = 0u;
        if (tid == 0) {
            sel[0] = kNone;
            sel[1] = 0u;
            if (level == 0) sel[2] = 0u;
        }
        __syncthreads();

        // Level 0 counts 0.0 entries and bins every entry; later levels bin
        // the entries whose higher bits equal the selected prefix.
        uint32_t nz = 0;
        auto visit = [&](uint32_t u) {
            const uint32_t key = order_key(u);
            if (level == 0) {
                nz += (u & 0x7FFFFFFFu) == 0u;
                if (has_boundary) hist_inc(hist, key >> 21);
            } else if ((key >> (dsh + dbits)) == prefix) {
                hist_inc(hist, (key >> dsh) & dmask);
            }
        };
        if ((uint32_t)tid < head) visit(xs[tid]);
        for (uint32_t q = (uint32_t)tid; q < nq; q += 4u * THREADS) {
            uint4 v[4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
                v[t] = q + t * THREADS < nq ? __ldg(xq + q + t * THREADS) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (q + t * THREADS < nq) {
                    visit(v[t].x);
                    visit(v[t].y);
                    visit(v[t].z);
                    visit(v[t].w);
                }
            }
        }
        if (tail0 + (uint32_t)tid < L) visit(xs[tail0 + tid]);
        if (level == 0) {
            nz = __reduce_add_sync(kFull, nz);
            if (lane == 0 && nz) atomicAdd(&sel[2], nz);
        }
        __syncthreads();
        if (!has_boundary) break;

        // The bin where the count from the top first reaches r; thread t
        // holds bins kBins-1-BPT*t down to kBins-BPT*(t+1).
        uint32_t h[BPT], sum = 0;
#pragma unroll
        for (int i = 0; i < BPT; ++i) {
            h[i] = hist[kBins - 1 - (BPT * tid + i)];
            sum += h[i];
        }
        uint32_t run = block_incl_scan<THREADS>(sum, scan) - sum;
#pragma unroll
        for (int i = 0; i < BPT; ++i) {
            if (run < r && run + h[i] >= r) {
                sel[0] = (uint32_t)(kBins - 1 - (BPT * tid + i));
                sel[1] = run;
            }
            run += h[i];
        }
        __syncthreads();
        const uint32_t d = sel[0];
        if (d == kNone) {   // cannot happen: the selected bin always holds >= r entries
            if (tid == 0) {
                atomicOr(&g_status, TOPK_DEV_INTERNAL);
                out[row] = res;
            }
            return;
        }
        above += sel[1];
        r -= sel[1];
        prefix = (prefix << dbits) | d;
        if (level == 2) tie = hist[d];
        __syncthreads();   // every thread has read sel and hist
    }
    if (tid == 0) {
        res.len = L;
        res.n_zero = sel[2];
        if (has_boundary) {
            const uint32_t T = prefix;   // the k-th key
            res.boundary_bits = key_bits(T);
            res.tie = tie;
            res.above = above;
            res.flags = TOPK_STAT_HAS_BOUNDARY;
            if (tie > 1u && above + tie > (uint32_t)k) res.flags |= TOPK_STAT_STRADDLE;
            if ((res.boundary_bits & 0x7FFFFFFFu) == 0u) res.flags |= TOPK_STAT_ZERO_BOUND;
        } else {
            res.above = L;
        }
        out[row] = res;
    }
}

#include "indexer_scores.cuh"

// Score array of topk_ragged_indexer_static: the chain's intermediate scores
// for callers that cannot allocate device memory.  The host passes its
// device address (looked up once per device) to the same two launches that
// topk_ragged_indexer makes; no kernel names it directly.
static __device__ __align__(256) float g_static_scores[TOPK_RAGGED_STATIC_SCORES];

// ------------------------------------------------------------------------- //
// Host side.
// ------------------------------------------------------------------------- //
typedef void (*KernelFn)(const Params);

// The top-k kernel of each planner variant (topk_plan::kRowKernel,
// kCluster512, kCluster1024).
const KernelFn kVariantFn[topk_plan::kVariants] = {
    topk_row_kernel<256>,
    topk_cluster_kernel<512>,
    topk_cluster_kernel<1024>,
};

struct DeviceInfo {
    bool ready = false;
    int status = TOPK_OK;
    topk_plan::DeviceShape shape = {};
};

std::mutex g_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;   // the driver's TMA descriptor encoder

// A TMA map over rows of 128 bf16 (256 bytes each): boxes of 64 columns
// (128 bytes, the 128-byte swizzle span) by box_rows rows.
bool encode_bf16_rows(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows)
{
    const cuuint64_t dims[2] = {(cuuint64_t)kIxDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kIxDim * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                          elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
DeviceInfo g_devices[kMaxDevices];
// Device address of g_static_scores on each device (null until the first
// topk_ragged_indexer_static call there looks it up).
float *g_static_scores_addr[kMaxDevices] = {};

using topk_plan::Plan;

Plan make_plan(int64_t n_scores, int32_t B, int32_t k, const DeviceInfo &dev)
{
    return topk_plan::make_plan(n_scores, B, k, dev.shape);
}

int init_locked(int device)
{
    DeviceInfo &d = g_devices[device];
    if (d.ready) return d.status;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return TOPK_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
        return TOPK_ERR_CUDA;
    if (major != 10 || minor != 3) {
        d.ready = true;
        d.status = TOPK_ERR_UNSUPPORTED_DEVICE;
        return d.status;
    }
    if (cudaSetDevice(device) != cudaSuccess) return TOPK_ERR_CUDA;
    int rc = TOPK_OK;
    topk_plan::DeviceShape &sh = d.shape;
    if (cudaDeviceGetAttribute(&sh.sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sh.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
        rc = TOPK_ERR_CUDA;
    if (rc == TOPK_OK &&
        cudaDeviceGetAttribute(&sh.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess)
        rc = TOPK_ERR_CUDA;
    for (int v = 0; v < topk_plan::kVariants && rc == TOPK_OK; ++v) {
        if (cudaFuncSetAttribute((const void *)kVariantFn[v], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 sh.max_smem) != cudaSuccess)
            rc = TOPK_ERR_CUDA;
        if (v != topk_plan::kRowKernel &&
            cudaFuncSetAttribute((const void *)kVariantFn[v], cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess)
            rc = TOPK_ERR_CUDA;
    }
    if (rc == TOPK_OK && cudaFuncSetAttribute((const void *)topk_stats_cluster_kernel<kStatsThreads>,
                                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        rc = TOPK_ERR_CUDA;
    if (rc == TOPK_OK && (cudaFuncSetAttribute((const void *)indexer_scores_kernel<1>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)IxCfg<1>::kSmemBytes) != cudaSuccess ||
                          cudaFuncSetAttribute((const void *)indexer_scores_kernel<kIxGroup>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)IxCfg<kIxGroup>::kSmemBytes) != cudaSuccess))
        rc = TOPK_ERR_CUDA;
    if (rc == TOPK_OK && !g_encode_tiled) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            rc = TOPK_ERR_CUDA;
        else
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    // Which cluster sizes each clustered variant can actually co-schedule
    // with the shared memory the planner gives it.
    for (int vi = topk_plan::kCluster512; vi < topk_plan::kVariants && rc == TOPK_OK; ++vi) {
        const int smem = topk_plan::variant_budget(sh, vi);
        for (int c = 2; c <= 16; c *= 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(c * 8), 1, 1);
            cfg.blockDim = dim3((unsigned)topk_plan::kVariantThreads[vi], 1, 1);
            cfg.dynamicSmemBytes = (size_t)smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, (const void *)kVariantFn[vi], &cfg) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            sh.max_clusters[vi][c] = n;
        }
        sh.max_clusters[vi][1] = 1;
    }
    cudaSetDevice(prev);
    if (rc == TOPK_OK) {
        d.ready = true;
        d.status = TOPK_OK;
    } else {
        cudaGetLastError();
    }
    return rc;
}

int ensure_init(int device, bool may_init)
{
    if (device < 0 || device >= kMaxDevices) return TOPK_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_devices[device].ready) return g_devices[device].status;
    if (!may_init) return TOPK_ERR_NOT_INITIALIZED;
    return init_locked(device);
}

}  // namespace

extern "C" {

int topk_ragged_abi_version(void) { return TOPK_RAGGED_ABI_VERSION; }

const char *topk_ragged_strerror(int status)
{
    switch (status) {
    case TOPK_OK: return "ok";
    case TOPK_ERR_INVALID_ARG: return "invalid argument";
    case TOPK_ERR_NOT_INITIALIZED: return "device not initialized (call topk_ragged_init outside stream capture)";
    case TOPK_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case TOPK_ERR_CUDA: return "CUDA runtime error";
    case TOPK_ERR_SCRATCH_TOO_SMALL:
        return "n_scores exceeds the library's fixed score array (TOPK_RAGGED_STATIC_SCORES)";
    default: return "unknown status";
    }
}

int topk_ragged_init(int device)
{
    if (device < 0 || device >= kMaxDevices) return TOPK_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    return init_locked(device);
}

static int validate(const float *scores, int64_t n_scores, const int32_t *row_starts,
                    const int32_t *lengths, int32_t B, int32_t k, int32_t offset_mode,
                    const int32_t *out_idx)
{
    if (k < 1 || k > TOPK_RAGGED_MAX_K || B < 0) return TOPK_ERR_INVALID_ARG;
    if ((int64_t)B * (int64_t)k >= ((int64_t)1 << 31)) return TOPK_ERR_INVALID_ARG;
    if ((offset_mode & ~(TOPK_OFFSET_ROW_START | TOPK_EXCLUDE_NEG_INF)) != 0) return TOPK_ERR_INVALID_ARG;
    if (n_scores < 0 || n_scores >= ((int64_t)1 << 31)) return TOPK_ERR_INVALID_ARG;
    if (B == 0) return TOPK_OK;
    if (!row_starts || !lengths || !out_idx) return TOPK_ERR_INVALID_ARG;
    if (!scores && n_scores > 0) return TOPK_ERR_INVALID_ARG;
    if (((uintptr_t)scores & 3u) != 0) return TOPK_ERR_INVALID_ARG;
    return TOPK_OK;
}

int topk_ragged_launch_info(int64_t n_scores, int32_t B, int32_t k, topk_launch_info *info)
{
    if (!info || k < 1 || k > TOPK_RAGGED_MAX_K || B < 0 || n_scores < 0) return TOPK_ERR_INVALID_ARG;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return TOPK_ERR_CUDA;
    int rc = ensure_init(device, true);
    if (rc != TOPK_OK) return rc;
    const Plan pl = make_plan(n_scores, B, k, g_devices[device]);
    info->threads = topk_plan::kVariantThreads[pl.variant];
    info->cluster = pl.cluster;
    info->stage_cap = pl.stage_cap;
    info->smem_bytes = pl.smem;
    info->grid = B > 0 ? pl.grid : 0;
    info->launches = B > 0 ? 1 : 0;
    return TOPK_OK;
}

static int launch(const float *scores, int64_t n_scores, const int32_t *row_starts, const int32_t *lengths,
                  int32_t B, int32_t k, int32_t offset_mode, const int32_t *page_table, int64_t pt_stride,
                  int32_t page_size, int32_t *out_idx, float *out_val, void *stream)
{
    cudaStream_t st = (cudaStream_t)stream;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return TOPK_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return TOPK_ERR_CUDA;
    int rc = ensure_init(device, cap == cudaStreamCaptureStatusNone);
    if (rc != TOPK_OK) return rc;
    const Plan pl = make_plan(n_scores, B, k, g_devices[device]);

    Params prm;
    prm.scores = scores;
    prm.n_scores = n_scores;
    prm.row_starts = row_starts;
    prm.lengths = lengths;
    prm.out_idx = out_idx;
    prm.out_val = out_val;
    prm.B = B;
    prm.k = k;
    prm.offset_mode = offset_mode;
    prm.stage_cap = pl.stage_cap;
    prm.win_cap = pl.win_cap;
    prm.off_win = pl.off_win;
    prm.off_keys = pl.off_keys;
    prm.page_table = page_table;
    prm.pt_stride = pt_stride;
    prm.page_size = page_size;
    const bool clustered = pl.variant != topk_plan::kRowKernel;
    prm.ahead = clustered ? 0 : g_devices[device].shape.sm_count * topk_plan::kRowCtasPerSm;
    prm.page_shift = (page_size & (page_size - 1)) == 0 ? __builtin_ctz((unsigned)page_size) : -1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
    cfg.blockDim = dim3((unsigned)topk_plan::kVariantThreads[pl.variant], 1, 1);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (clustered) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)pl.cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    if (cudaLaunchKernelEx(&cfg, kVariantFn[pl.variant], prm) != cudaSuccess) {
        cudaGetLastError();
        return TOPK_ERR_CUDA;
    }
    return TOPK_OK;
}

int topk_ragged(const float *scores, int64_t n_scores, const int32_t *row_starts,
                const int32_t *lengths, int32_t B, int32_t k, int32_t offset_mode,
                int32_t *out_idx, float *out_val, void *stream)
{
    const int rc = validate(scores, n_scores, row_starts, lengths, B, k, offset_mode, out_idx);
    if (rc != TOPK_OK || B == 0) return rc;
    return launch(scores, n_scores, row_starts, lengths, B, k, offset_mode, nullptr, 0, 1, out_idx, out_val,
                  stream);
}

int topk_ragged_paged(const float *scores, int64_t n_scores, const int32_t *row_starts,
                      const int32_t *lengths, int32_t B, int32_t k, int32_t flags,
                      const int32_t *page_table, int64_t page_table_stride, int32_t page_size,
                      int32_t *out_idx, float *out_val, void *stream)
{
    if ((flags & ~TOPK_EXCLUDE_NEG_INF) != 0 || page_size < 1 || page_table_stride < 0)
        return TOPK_ERR_INVALID_ARG;
    const int rc = validate(scores, n_scores, row_starts, lengths, B, k, flags, out_idx);
    if (rc != TOPK_OK || B == 0) return rc;
    if (!page_table) return TOPK_ERR_INVALID_ARG;
    return launch(scores, n_scores, row_starts, lengths, B, k, flags, page_table, page_table_stride, page_size,
                  out_idx, out_val, stream);
}

int topk_ragged_stats(const float *scores, int64_t n_scores, const int32_t *row_starts,
                      const int32_t *lengths, int32_t B, int32_t k, topk_row_stats *out,
                      void *stream)
{
    if (k < 1 || k > TOPK_RAGGED_MAX_K || B < 0) return TOPK_ERR_INVALID_ARG;
    if (n_scores < 0 || n_scores >= ((int64_t)1 << 31)) return TOPK_ERR_INVALID_ARG;
    if (B == 0) return TOPK_OK;
    if (!row_starts || !lengths || !out) return TOPK_ERR_INVALID_ARG;
    if (!scores && n_scores > 0) return TOPK_ERR_INVALID_ARG;
    if (((uintptr_t)scores & 3u) != 0) return TOPK_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return TOPK_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return TOPK_ERR_CUDA;
    const int rc = ensure_init(device, cap == cudaStreamCaptureStatusNone);
    if (rc != TOPK_OK) return rc;
    // One cluster per row: a batch of few, long rows splits each row over up
    // to 16 CTAs, so that the batch covers about two CTAs per SM and every
    // CTA keeps at least 16 K scores on average; otherwise one CTA per row.
    int cs = 1;
    while (cs < 16 && (int64_t)B * cs * 2 <= 2LL * g_devices[device].shape.sm_count &&
           n_scores >= (int64_t)B * cs * 2 * 16384)
        cs *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)B * cs), 1, 1);
    cfg.blockDim = dim3((unsigned)kStatsThreads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cs;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cs == 1) cfg.numAttrs = 1;   // no cluster
    const cudaError_t err =
        cs == 1 ? cudaLaunchKernelEx(&cfg, topk_stats_kernel<kStatsThreads>, scores, n_scores, row_starts, lengths,
                                     k, out)
                : cudaLaunchKernelEx(&cfg, topk_stats_cluster_kernel<kStatsThreads>, scores, n_scores, row_starts,
                                     lengths, k, out);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return TOPK_ERR_CUDA;
    }
    return TOPK_OK;
}

int topk_ragged_indexer_scores(const uint16_t *q, const float *w, const float *bias, const uint16_t *keys,
                               int64_t n_keys, const int32_t *key_starts, const int32_t *lengths,
                               const int32_t *score_starts, int32_t B, float scale, float *scores, int64_t n_scores,
                               void *stream)
{
    // n_keys leaves room for a last partial tile's row coordinate in int32.
    if (B < 0 || n_keys < 1 || n_keys > ((int64_t)1 << 31) - kIxTile || n_scores < 0 ||
        n_scores >= ((int64_t)1 << 31))
        return TOPK_ERR_INVALID_ARG;
    if ((int64_t)B * kIxHeads >= ((int64_t)1 << 31) || !(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
        return TOPK_ERR_INVALID_ARG;
    if (B == 0) return TOPK_OK;
    if (!q || !w || !keys || !key_starts || !lengths || !score_starts || (!scores && n_scores > 0))
        return TOPK_ERR_INVALID_ARG;
    if (((uintptr_t)q & 15u) || ((uintptr_t)keys & 15u) || ((uintptr_t)w & 15u) || ((uintptr_t)bias & 3u) ||
        ((uintptr_t)scores & 3u))
        return TOPK_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return TOPK_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return TOPK_ERR_CUDA;
    const int rc = ensure_init(device, cap == cudaStreamCaptureStatusNone);
    if (rc != TOPK_OK) return rc;
    // Rows share key tiles only when the key buffer is read by more than one
    // row on average (a causal prefill chunk); otherwise the single-row
    // instance keeps a deeper ring for the key stream.  Either is correct.
    const bool grouped = 2 * n_keys <= n_scores;
    CUtensorMap tmap_k, tmap_q;
    if (!encode_bf16_rows(&tmap_k, keys, (uint64_t)n_keys, kIxTile) ||
        !encode_bf16_rows(&tmap_q, q, (uint64_t)B * kIxHeads, grouped ? IxCfg<kIxGroup>::kQRows : IxCfg<1>::kQRows))
        return TOPK_ERR_INVALID_ARG;
    IxParams prm;
    prm.w = w;
    prm.bias = bias;
    prm.key_starts = key_starts;
    prm.lengths = lengths;
    prm.score_starts = score_starts;
    prm.scores = scores;
    prm.n_keys = n_keys;
    prm.n_scores = n_scores;
    prm.B = B;
    prm.scale = scale;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)g_devices[device].shape.sm_count, 1, 1);
    cfg.blockDim = dim3((unsigned)(grouped ? IxCfg<kIxGroup>::kThreads : IxCfg<1>::kThreads), 1, 1);
    cfg.dynamicSmemBytes = grouped ? IxCfg<kIxGroup>::kSmemBytes : IxCfg<1>::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = grouped ? cudaLaunchKernelEx(&cfg, indexer_scores_kernel<kIxGroup>, tmap_k, tmap_q, prm)
                                    : cudaLaunchKernelEx(&cfg, indexer_scores_kernel<1>, tmap_k, tmap_q, prm);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return TOPK_ERR_CUDA;
    }
    return TOPK_OK;
}

int topk_ragged_indexer(const uint16_t *q, const float *w, const float *bias, const uint16_t *keys, int64_t n_keys,
                        const int32_t *key_starts, const int32_t *lengths, const int32_t *score_starts, int32_t B,
                        float scale, float *scores, int64_t n_scores, int32_t k, int32_t flags, int32_t *out_idx,
                        float *out_val, void *stream)
{
    if ((flags & ~TOPK_EXCLUDE_NEG_INF) != 0) return TOPK_ERR_INVALID_ARG;
    int rc = validate(scores, n_scores, score_starts, lengths, B, k, flags, out_idx);
    if (rc != TOPK_OK || B == 0) return rc;
    rc = topk_ragged_indexer_scores(q, w, bias, keys, n_keys, key_starts, lengths, score_starts, B, scale, scores,
                                    n_scores, stream);
    if (rc != TOPK_OK) return rc;
    return topk_ragged(scores, n_scores, score_starts, lengths, B, k, flags, out_idx, out_val, stream);
}

int topk_ragged_indexer_static(const uint16_t *q, const float *w, const float *bias, const uint16_t *keys,
                               int64_t n_keys, const int32_t *key_starts, const int32_t *lengths,
                               const int32_t *score_starts, int32_t B, float scale, int64_t n_scores, int32_t k,
                               int32_t flags, int32_t *out_idx, float *out_val, void *stream)
{
    if (n_scores > (int64_t)TOPK_RAGGED_STATIC_SCORES) return TOPK_ERR_SCRATCH_TOO_SMALL;
    if (n_scores < 0 || k < 1 || k > TOPK_RAGGED_MAX_K || B < 0 || (flags & ~TOPK_EXCLUDE_NEG_INF) != 0)
        return TOPK_ERR_INVALID_ARG;
    if (B == 0) return TOPK_OK;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return TOPK_ERR_CUDA;
    if (device < 0 || device >= kMaxDevices) return TOPK_ERR_UNSUPPORTED_DEVICE;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing((cudaStream_t)stream, &cap) != cudaSuccess) return TOPK_ERR_CUDA;
    float *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        scratch = g_static_scores_addr[device];
        if (!scratch) {
            if (cap != cudaStreamCaptureStatusNone) return TOPK_ERR_NOT_INITIALIZED;
            // Set-up, once per device, with that device current: in host code
            // g_static_scores names a host-side stand-in, not device memory.
            if (cudaGetSymbolAddress((void **)&scratch, g_static_scores) != cudaSuccess || !scratch) {
                cudaGetLastError();
                return TOPK_ERR_CUDA;
            }
            g_static_scores_addr[device] = scratch;
        }
    }
    return topk_ragged_indexer(q, w, bias, keys, n_keys, key_starts, lengths, score_starts, B, scale, scratch,
                               n_scores, k, flags, out_idx, out_val, stream);
}

int topk_ragged_wait_probe(uint32_t polls, void *stream)
{
    if (polls == 0 || polls > kWaitLimit) return TOPK_ERR_INVALID_ARG;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return TOPK_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing((cudaStream_t)stream, &cap) != cudaSuccess) return TOPK_ERR_CUDA;
    const int rc = ensure_init(device, cap == cudaStreamCaptureStatusNone);
    if (rc != TOPK_OK) return rc;
    wait_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(polls);
    return cudaPeekAtLastError() == cudaSuccess ? TOPK_OK : (cudaGetLastError(), TOPK_ERR_CUDA);
}

int topk_ragged_device_status(uint32_t *host_out, void *stream)
{
    if (!host_out) return TOPK_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status) != cudaSuccess) return TOPK_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, addr, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemsetAsync(addr, 0, sizeof(uint32_t), st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return TOPK_ERR_CUDA;
    }
    *host_out = v;
    return TOPK_OK;
}

}  // extern "C"
