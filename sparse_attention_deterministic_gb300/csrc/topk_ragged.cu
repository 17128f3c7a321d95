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
//   * one row per thread-block cluster of C CTAs (C = 1..16, chosen from B
//     on the host); each CTA owns a contiguous, 16-byte-aligned slice of the
//     row and keeps as much of it as fits in shared memory, so the row is
//     read from HBM once; the rest of a very long slice is re-read from L2;
//   * an MSB-first radix select on the monotone uint32 order key with digits
//     of 11, 11 and 10 bits; per-CTA histograms use shared-memory atomics
//     (colliding lanes are merged by the hardware) and are merged into the cluster
//     leader through distributed shared memory (red.shared::cluster), so the
//     k-th key T, the count above it and the count needed from its tie set
//     are exact integers, independent of scheduling;
//   * every entry above T is a winner; entries equal to T are ranked by
//     index with ordered per-warp / per-CTA prefix counts (the tie set is
//     taken in index order, so its first r members are the smallest indices,
//     and they already sit in canonical order after the winners);
//   * the winners (fewer than k) are gathered into the leader as unique
//     (key << 32 | ~index) composites and sorted descending in shared
//     memory; the row is written with coalesced stores.
//
// Nothing is allocated; the only global state is a status word for data
// errors.  All cross-CTA synchronisation uses hardware cluster barriers.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "topk_ragged.h"

namespace {

constexpr int kBins = 2048;            // 11-bit digits (the last level uses 10 bits)
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
    int32_t grouped;     // clusters take groups of rows (see assign_rows)
};

// Per-CTA control block at the start of dynamic shared memory.
struct __align__(16) Ctrl {
    uint32_t sel_digit;  // result of the last threshold search
    uint32_t sel_gt;     //   entries above the chosen bin (within the prefix)
    uint32_t sel_cnt;    //   entries in the chosen bin
    uint32_t sel_done;   //   1: the k-th key is +0.0 (plateau shortcut)
    uint32_t zeros;      // this CTA's count of exact +0.0 scores
    uint32_t zeros_tot;  // leader: the cluster's count of exact +0.0 scores
    uint32_t win_count;  // leader: winner slots handed out
    uint32_t pad;
    uint32_t kmax;       // this CTA's largest order key
    uint32_t kmax_tot;   // leader: the cluster's largest order key
    uint32_t wmin;       // leader: the smallest winner key
    uint32_t pad2;
    uint32_t warp_zeros[32];
    uint32_t warp_ties[32];
    uint32_t scan[36];
    uint64_t scan64[32];
};

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

__device__ __forceinline__ void dsmem_red_add(uint32_t addr, uint32_t v)
{
    asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t dsmem_atom_add(uint32_t addr, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void dsmem_st64(uint32_t addr, uint64_t v)
{
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ void dsmem_red_max(uint32_t addr, uint32_t v)
{
    asm volatile("red.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void dsmem_red_min(uint32_t addr, uint32_t v)
{
    asm volatile("red.shared::cluster.min.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t dsmem_ld(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void dsmem_st(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
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

// Histogram increment.  On this GPU a shared-memory atomic add whose lanes
// collide on one address is merged by the hardware at full rate, while
// __match_any_sync is serialised per distinct value, so the plain per-lane
// atomic is the cheapest form on every digit distribution, plateau included.
__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t digit, bool valid)
{
    if (valid) atomicAdd(&hist[digit], 1u);
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
// network instead.  b[] is scratch for n composites, cur[] kBins words.
// ------------------------------------------------------------------------- //
template <int THREADS>
__device__ void sort_and_write(uint64_t *a, uint64_t *b, int n, int cap_pow2, uint32_t kmin,
                               uint32_t kmax, uint32_t *cur, uint64_t *sm64, int32_t *oi, float *ov,
                               int64_t idx_offset)
{
    constexpr int BPT = kBins / THREADS;
    const int tid = threadIdx.x;
    const uint32_t range = kmax - kmin;
    const int s = max(0, (32 - __clz(range)) - 11);
    for (int i = tid; i < kBins; i += THREADS) cur[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += THREADS) atomicAdd(&cur[((uint32_t)(a[i] >> 32) - kmin) >> s], 1u);
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
        for (int p = tid; p < n; p += THREADS) {
            const uint64_t c = a[p];
            oi[p] = (int32_t)(idx_offset + (int32_t)(~(uint32_t)c));
            if (ov) ov[p] = __uint_as_float(key_bits((uint32_t)(c >> 32)));
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
        oi[pos] = (int32_t)(idx_offset + (int32_t)(~(uint32_t)x));
        if (ov) ov[pos] = __uint_as_float(key_bits((uint32_t)(x >> 32)));
    }
}

__device__ __forceinline__ void pad_out(int32_t *oi, float *ov, int from, int to)
{
    for (int p = from + (int)threadIdx.x; p < to; p += (int)blockDim.x) {
        oi[p] = -1;
        if (ov) ov[p] = __uint_as_float(kNegInfBits);
    }
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
    const int B = p.B;
    const int G = (int)(gridDim.x / csize), cid = (int)(blockIdx.x / csize);
    uint32_t *eff = scratch;              // B valid lengths (0: nothing to select)
    uint32_t *by_rank = scratch + 1024;   // row index of every rank
    for (int i = tid; i < B; i += THREADS) {
        int64_t len;
        eff[i] = row_window_ok(p, i, len) ? (uint32_t)len : 0u;
    }
    __syncthreads();
    for (int i = tid; i < B; i += THREADS) {
        const uint32_t e = eff[i];
        int rank = 0;
        for (int j = 0; j < B; ++j) {
            const uint32_t ej = eff[j];
            rank += (ej > e) || (ej == e && j < i);
        }
        by_rank[rank] = (uint32_t)i;
    }
    __syncthreads();
    if (tid == 0) {
        int rows[16];
        uint32_t len[16];
        int m = 0;
        for (int t0 = 0; t0 < B; t0 += 2 * G) {
            const int ta = t0 + cid, tb = t0 + 2 * G - 1 - cid;
            if (ta < B && m < 16) { rows[m] = (int)by_rank[ta]; len[m] = eff[rows[m]]; ++m; }
            if (tb < B && m < 16) { rows[m] = (int)by_rank[tb]; len[m] = eff[rows[m]]; ++m; }
        }
        // Rows are listed in rank order, so the rows with work come first.
        int mv = 0;
        uint64_t E = 0;
        while (mv < m && len[mv] > 0) E += len[mv++];
        int mine = -1;
        uint32_t g0 = 0, gsize = 0;
        if (mv > 0) {
            uint32_t c[16];
            uint32_t used = 0;
            const uint32_t spare = csize - (uint32_t)mv;
            for (int i = 0; i < mv; ++i) {
                c[i] = 1u + (uint32_t)((uint64_t)spare * len[i] / E);
                used += c[i];
            }
            for (int i = 0; used < csize; i = (i + 1) % mv) {
                ++c[i];
                ++used;
            }
            uint32_t start = 0;
            for (int i = 0; i < mv; ++i) {
                if (crank >= start && crank < start + c[i]) {
                    mine = rows[i];
                    g0 = start;
                    gsize = c[i];
                }
                start += c[i];
            }
        }
        slot[0] = (uint32_t)mine;
        slot[1] = g0;
        slot[2] = gsize;
        // The cluster's first CTA pads the rows with nothing to select.
        slot[3] = (uint32_t)(m - mv);
        for (int i = mv; i < m; ++i) slot[4 + i - mv] = (uint32_t)rows[i];
    }
    __syncthreads();
    RowGroup g;
    g.row = (int)slot[0];
    g.g0 = slot[1];
    g.gsize = slot[2];
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
// The kernel.  CLUSTER = false: one row per CTA.  CLUSTER = true: each
// cluster takes a group of rows (assign_rows) and every row is worked on by
// a contiguous group of the cluster's CTAs; the group's first CTA is the
// row's leader (cluster-wide histograms, threshold search, winner list,
// sort).  With one row per cluster the group is the whole cluster.
//
// Every pass over a CTA's slice walks the same contiguous per-warp
// segments, U quads per lane in flight, so per-warp counts taken in one pass
// give index-ordered positions in a later one.
// ------------------------------------------------------------------------- //
template <int THREADS, bool CLUSTER>
__global__ void __launch_bounds__(THREADS, 2048 / THREADS / 2) topk_ragged_kernel(const Params p)
{
    constexpr int NW = THREADS / 32;
    constexpr int U = 4;                       // quads in flight per lane
    constexpr uint32_t kZeroKey = 0x80000000u; // order key of +0.0
    constexpr uint32_t kZeroDigit = kZeroKey >> 21;
    extern __shared__ __align__(16) unsigned char smem[];
    Ctrl &ctrl = *reinterpret_cast<Ctrl *>(smem);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + sizeof(Ctrl));
    uint32_t *hist_tot = hist + kBins;   // the row leader's group-wide histogram (CLUSTER only)
    uint64_t *win = reinterpret_cast<uint64_t *>(smem + p.off_win);
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + p.off_keys);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int row;
    uint32_t grank = 0, gsize = 1, g0 = 0;
    if (CLUSTER) {
        const uint32_t crank = cluster_rank(), csize = cluster_size();
        if (p.grouped) {
            const RowGroup g = assign_rows<THREADS>(p, crank, csize, hist, ctrl.scan);
            if (g.row < 0) return;   // uniform over the cluster: nothing to select
            row = g.row;
            g0 = g.g0;
            gsize = g.gsize;
            grank = crank - g0;
        } else {
            row = (int)(blockIdx.x / csize);
            gsize = csize;
            grank = crank;
        }
    } else {
        row = (int)blockIdx.x;
    }
    const bool leader = grank == 0;

    // ---- a1: metadata, window checks ----------------------------------- //
    const int64_t rs = p.row_starts[row];
    int64_t len = p.lengths[row];
    if (len < 0) len = 0;
    uint32_t bad = 0;
    if (len >= (int64_t)TOPK_RAGGED_MAX_LEN)
        bad = TOPK_DEV_LEN_ENVELOPE;
    else if (rs < 0 || rs + len > p.n_scores)
        bad = TOPK_DEV_BAD_WINDOW;
    int32_t *oi = p.out_idx + (int64_t)row * p.k;
    float *ov = p.out_val ? p.out_val + (int64_t)row * p.k : nullptr;
    if (bad || len == 0) {
        // Grouped clusters never get here (such rows are padded above); with
        // one row per cluster the decision is uniform over the cluster and
        // precedes every cluster barrier.
        if (leader) {
            if (bad && tid == 0) atomicOr(&g_status, bad);
            pad_out(oi, ov, 0, p.k);
        }
        return;
    }
    const int32_t L = (int32_t)len;
    const uint32_t k_eff = (uint32_t)(p.k < L ? p.k : L);
    const int64_t idx_offset = p.offset_mode == TOPK_OFFSET_ROW_START ? rs : 0;

    // ---- slice of this CTA (16-byte aligned body split by quads) ----------- //
    Slice s;
    {
        const uint64_t pa = (uint64_t)(uintptr_t)p.scores >> 2;   // element address
        const int64_t e0 = rs, e1 = rs + L;
        int64_t a0 = e0 + (int64_t)((4u - (uint32_t)((pa + (uint64_t)e0) & 3u)) & 3u);
        if (a0 > e1) a0 = e1;
        const int64_t n4 = (e1 - a0) >> 2;
        const int64_t qlo = n4 * grank / gsize, qhi = n4 * (grank + 1) / gsize;
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
    const WarpSeg seg = warp_segment<THREADS>(s.nq, warp);

    // ---- init shared state ------------------------------------------------ //
    for (int b = tid; b < kBins; b += THREADS) {
        hist[b] = 0u;
        if (CLUSTER && leader) hist_tot[b] = 0u;
    }
    if (tid == 0) {
        ctrl.sel_digit = 0u;
        ctrl.sel_gt = 0u;
        ctrl.sel_cnt = 0u;
        ctrl.sel_done = 0u;
        ctrl.zeros = 0u;
        ctrl.zeros_tot = 0u;
        ctrl.win_count = 0u;
        ctrl.kmax = 0u;
        ctrl.kmax_tot = 0u;
        ctrl.wmin = kFull;
    }
    __syncthreads();
    if (CLUSTER) cluster_arrive();   // B0: every CTA started and zeroed (waited before the flush)

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

    const uint32_t lead_hist_tot = CLUSTER ? dsmem_addr(hist_tot, g0) : 0u;

    // Running selection state (identical in every thread of the group).
    uint32_t prefix = 0, n_gt = 0, r = k_eff, cnt = 0;
    bool plateau = false;   // T is +0.0, found from the zero count
    bool sel_done = false;  // the k-th key is known

    // ---- a4+a5: radix levels of 11, 11 and 10 bits.  In a cluster every
    //      CTA runs all three levels' barriers, working or not, because the
    //      cluster's rows may finish at different levels. --------------- //
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
        const uint32_t *htot = hist;
        if (CLUSTER) {
            if (level == 0) cluster_wait();   // B0 complete: the leaders' totals are zeroed
            if (!sel_done) {
                for (int b = tid; b < kBins; b += THREADS) {
                    const uint32_t v = hist[b];
                    if (v) dsmem_red_add(lead_hist_tot + 4u * (uint32_t)b, v);
                }
                if (level == 0 && tid == 0) {
                    if (ctrl.zeros) dsmem_red_add(dsmem_addr(&ctrl.zeros_tot, g0), ctrl.zeros);
                    dsmem_red_max(dsmem_addr(&ctrl.kmax_tot, g0), ctrl.kmax);
                }
            }
            cluster_sync();   // B1: each leader holds its group's histogram
            htot = hist_tot;
        }
        if ((!CLUSTER || leader) && !sel_done) {
            if (find_bin<THREADS>(htot, r, ctrl.scan, d, gt, c)) {
                // Plateau shortcut: the boundary bin holds only exact +0.0, so
                // the k-th key is +0.0 and the finer levels are not needed.
                const uint32_t ztot = CLUSTER ? ctrl.zeros_tot : ctrl.zeros;
                const uint32_t done = (level == 0 && d == kZeroDigit && c == ztot) ? 1u : 0u;
                if (CLUSTER) {
                    for (uint32_t rk = g0; rk < g0 + gsize; ++rk) {
                        dsmem_st(dsmem_addr(&ctrl.sel_digit, rk), d);
                        dsmem_st(dsmem_addr(&ctrl.sel_gt, rk), gt);
                        dsmem_st(dsmem_addr(&ctrl.sel_cnt, rk), c);
                        dsmem_st(dsmem_addr(&ctrl.sel_done, rk), done);
                    }
                } else {
                    ctrl.sel_digit = d;
                    ctrl.sel_gt = gt;
                    ctrl.sel_cnt = c;
                    ctrl.sel_done = done;
                }
            }
        }
        if (CLUSTER) {
            if (leader && !sel_done) {
                __syncthreads();
                for (int b = tid; b < kBins; b += THREADS) hist_tot[b] = 0u;
            }
            cluster_sync();   // B2: selections visible to every CTA of their group
        } else {
            __syncthreads();
        }
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
        if (!CLUSTER && sel_done) break;
    }
    const uint32_t T = prefix;   // exact k-th key; n_gt above it, take r of its cnt ties
    const uint32_t tval = key_bits(T);

    // ---- a6+a7: one pass over the slice.  Winners (key > T) go to the
    //      leader's list in any order (their composites are unique, the sort
    //      makes the order canonical).  Ties (key == T): the first r in
    //      group-wide index order go straight to positions n_gt + ordinal.
    //      On the plateau every tie is a +0.0 and the per-warp zero counts of
    //      the streaming pass already give each warp's first ordinal; else
    //      the pass counts ties per warp and a second pass writes them. --- //
    uint32_t tie_base = 0, local_eq = cnt;
    if (CLUSTER) {
        local_eq = plateau ? ctrl.zeros : hist[T & 0x3FFu];
        uint32_t part = 0;
        if (warp == 0 && lane < (int)grank) {
            const void *src = plateau ? (const void *)&ctrl.zeros : (const void *)&hist[T & 0x3FFu];
            part = dsmem_ld(dsmem_addr(src, g0 + (uint32_t)lane));
        }
        if (warp == 0) part = __reduce_add_sync(kFull, part);
        if (tid == 0) ctrl.scan[0] = part;
        __syncthreads();
        tie_base = ctrl.scan[0];
    }
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
    const uint32_t win_count_addr = CLUSTER ? dsmem_addr(&ctrl.win_count, g0) : 0u;
    const uint32_t win_addr = CLUSTER ? dsmem_addr(win, g0) : 0u;
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
                    base = CLUSTER ? dsmem_atom_add(win_count_addr, wtot) : atomicAdd(&ctrl.win_count, wtot);
                slot += __shfl_sync(kFull, base, 0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if ((wm >> i) & 1u) {
                        const uint32_t j = (uint32_t)(s.jbase + 4 * q + i);
                        const uint64_t comp = ((uint64_t)e[i] << 32) | (uint64_t)(~j);
                        wmin = min(wmin, e[i]);
                        if (slot < (uint32_t)p.win_cap) {
                            if (CLUSTER) dsmem_st64(win_addr + 8u * slot, comp);
                            else win[slot] = comp;
                        }
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
                                    oi[n_gt + tord] = (int32_t)(idx_offset + j);
                                    if (ov) ov[n_gt + tord] = __uint_as_float(tval);
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
    if (lane == 0 && wmin != kFull) {
        if (CLUSTER) dsmem_red_min(dsmem_addr(&ctrl.wmin, g0), wmin);
        else atomicMin(&ctrl.wmin, wmin);
    }

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
                                oi[n_gt + tord] = (int32_t)(idx_offset + j);
                                if (ov) ov[n_gt + tord] = __uint_as_float(tval);
                            }
                            ++tord;
                        }
                    }
                    trun += ttot;
                }
            }
        }
    }

    // ---- a8+a9: the leader sorts the winners and writes the row ----------- //
    if (CLUSTER) {
        cluster_sync();   // B3: every winner is in its leader's list
        if (!leader) return;
    } else {
        __syncthreads();
    }
    const uint32_t n_win = ctrl.win_count;
    if (n_win != n_gt || n_gt > (uint32_t)p.win_cap) {
        if (tid == 0) atomicOr(&g_status, TOPK_DEV_INTERNAL);
    }
    const uint32_t n_sort = n_gt < (uint32_t)p.win_cap ? n_gt : (uint32_t)p.win_cap;
    if (n_sort > 0) {
        const uint32_t kmax = CLUSTER ? ctrl.kmax_tot : ctrl.kmax;
        sort_and_write<THREADS>(win, reinterpret_cast<uint64_t *>(keys), (int)n_sort, p.win_cap,
                                ctrl.wmin, kmax, hist, ctrl.scan64, oi, ov, idx_offset);
    }
    pad_out(oi, ov, (int)k_eff, p.k);
}

// ------------------------------------------------------------------------- //
// Host side.
// ------------------------------------------------------------------------- //
typedef void (*KernelFn)(const Params);

struct Variant {
    KernelFn fn;
    int threads;
    bool cluster;
};

const Variant kVariants[] = {
    {topk_ragged_kernel<256, false>, 256, false},
    {topk_ragged_kernel<512, true>, 512, true},
    {topk_ragged_kernel<1024, true>, 1024, true},
};

struct DeviceInfo {
    bool ready = false;
    int status = TOPK_OK;
    int sm_count = 0;
    int max_smem = 0;      // opt-in dynamic shared memory per block
    int smem_per_sm = 0;   // shared memory per multiprocessor
    // max_clusters[variant][C]: co-resident clusters of C CTAs (0 = not launchable)
    int max_clusters[3][17] = {};
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

struct Plan {
    const Variant *v;
    int cluster;
    int grouped;
    int stage_cap;
    int win_cap;
    int off_win, off_keys, smem;
    int grid;
};

int next_pow2(int x)
{
    int n = 1;
    while (n < x) n <<= 1;
    return n;
}

int header_bytes(bool cluster)
{
    return (int)sizeof(Ctrl) + kBins * 4 * (cluster ? 2 : 1);
}

// Launch shape from the host arguments alone (row lengths live on the
// device and are never read here).
//   * B >= 4 x SMs: one 256-thread CTA per row, several CTAs per SM.
//   * B x 16 <= SMs: a 16-CTA cluster of 1024-thread CTAs per row, each CTA
//     with all of an SM's shared memory (very long rows stage the most).
//   * otherwise: one resident wave of G clusters of CS 512-thread CTAs (two
//     per SM); the clusters share out the rows by length and each cluster
//     deals its CTAs to its rows in proportion to their lengths
//     (assign_rows), so every CTA gets a similar slice.
//   * batches too large for that wave fall back to one CTA per row.
// Each CTA stages what shared memory allows and re-reads the rest of its
// slice from L2.
Plan make_plan(int32_t B, int32_t k, const DeviceInfo &dev)
{
    Plan pl{};
    pl.win_cap = next_pow2(k - 1 > 1 ? k - 1 : 1);
    const int sms = dev.sm_count;
    int vi = 0, cluster = 1, smem_budget = 0, grid = B;
    pl.grouped = 0;
    if (B < 4 * sms) {
        if ((int64_t)B * 16 <= sms && dev.max_clusters[2][16] > 0) {
            vi = 2;
            cluster = 16;
            smem_budget = dev.max_smem;
            grid = B * 16;
        } else {
            for (int cs = 16; cs >= 2; cs /= 2) {
                const int g = min(2 * sms / cs, dev.max_clusters[1][cs]);
                if (g > 0 && (int64_t)g * cs >= B) {
                    vi = 1;
                    cluster = cs;
                    smem_budget = dev.smem_per_sm / 2 - 1024;
                    grid = g * cs;
                    pl.grouped = 1;
                    break;
                }
            }
        }
    }
    pl.v = &kVariants[vi];
    pl.cluster = cluster;
    pl.off_win = header_bytes(pl.v->cluster);
    // The staged keys are read as 16-byte vectors: keep them 128-byte aligned
    // whatever the winner array's size (k <= 2 gives a single 8-byte slot).
    pl.off_keys = (pl.off_win + pl.win_cap * 8 + 127) & ~127;
    int stage_cap = smem_budget > 0 ? ((smem_budget - pl.off_keys) / 4) & ~127 : 4096 + 256;
    // The staging area doubles as the sort's second buffer after compaction.
    if (stage_cap < 2 * pl.win_cap) stage_cap = 2 * pl.win_cap;
    pl.stage_cap = stage_cap;
    pl.smem = pl.off_keys + stage_cap * 4;
    pl.grid = grid;
    return pl;
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
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
        rc = TOPK_ERR_CUDA;
    if (rc == TOPK_OK &&
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess)
        rc = TOPK_ERR_CUDA;
    for (const Variant &v : kVariants) {
        if (rc != TOPK_OK) break;
        if (cudaFuncSetAttribute((const void *)v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 d.max_smem) != cudaSuccess)
            rc = TOPK_ERR_CUDA;
        if (v.cluster && cudaFuncSetAttribute((const void *)v.fn,
                                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            rc = TOPK_ERR_CUDA;
    }
    // Which cluster sizes each clustered variant can actually co-schedule
    // with the shared memory the planner gives it.
    for (int vi = 1; vi < 3 && rc == TOPK_OK; ++vi) {
        const Variant &v = kVariants[vi];
        const int smem = vi == 2 ? d.max_smem : d.smem_per_sm / 2 - 1024;
        for (int c = 2; c <= 16; c *= 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(c * 8), 1, 1);
            cfg.blockDim = dim3((unsigned)v.threads, 1, 1);
            cfg.dynamicSmemBytes = (size_t)smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, (const void *)v.fn, &cfg) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            d.max_clusters[vi][c] = n;
        }
        d.max_clusters[vi][1] = 1;
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
    if (offset_mode != TOPK_OFFSET_ROW_LOCAL && offset_mode != TOPK_OFFSET_ROW_START)
        return TOPK_ERR_INVALID_ARG;
    if (n_scores < 0 || n_scores >= ((int64_t)1 << 31)) return TOPK_ERR_INVALID_ARG;
    if (B == 0) return TOPK_OK;
    if (!row_starts || !lengths || !out_idx) return TOPK_ERR_INVALID_ARG;
    if (!scores && n_scores > 0) return TOPK_ERR_INVALID_ARG;
    if (((uintptr_t)scores & 3u) != 0) return TOPK_ERR_INVALID_ARG;
    return TOPK_OK;
}

int topk_ragged_launch_info(int32_t B, int32_t k, topk_launch_info *info)
{
    if (!info || k < 1 || k > TOPK_RAGGED_MAX_K || B < 0) return TOPK_ERR_INVALID_ARG;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return TOPK_ERR_CUDA;
    int rc = ensure_init(device, true);
    if (rc != TOPK_OK) return rc;
    const Plan pl = make_plan(B, k, g_devices[device]);
    info->threads = pl.v->threads;
    info->cluster = pl.cluster;
    info->stage_cap = pl.stage_cap;
    info->smem_bytes = pl.smem;
    info->grid = B > 0 ? pl.grid : 0;
    info->launches = B > 0 ? 1 : 0;
    return TOPK_OK;
}

int topk_ragged(const float *scores, int64_t n_scores, const int32_t *row_starts,
                const int32_t *lengths, int32_t B, int32_t k, int32_t offset_mode,
                int32_t *out_idx, float *out_val, void *stream)
{
    int rc = validate(scores, n_scores, row_starts, lengths, B, k, offset_mode, out_idx);
    if (rc != TOPK_OK || B == 0) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return TOPK_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return TOPK_ERR_CUDA;
    rc = ensure_init(device, cap == cudaStreamCaptureStatusNone);
    if (rc != TOPK_OK) return rc;
    const Plan pl = make_plan(B, k, g_devices[device]);

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
    prm.grouped = pl.grouped;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid, 1, 1);
    cfg.blockDim = dim3((unsigned)pl.v->threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (pl.v->cluster) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)pl.cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&cfg, pl.v->fn, prm) != cudaSuccess) {
        cudaGetLastError();
        return TOPK_ERR_CUDA;
    }
    return TOPK_OK;
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
