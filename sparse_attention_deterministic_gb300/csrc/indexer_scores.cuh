// indexer_scores.cuh -- lightning-indexer scores on the tcgen05 tensor cores.
//
// Included by topk_ragged.cu inside its anonymous namespace (it shares that
// file's status word, mbarrier helpers and block scan).
//
// The scores are those of the DSA lightning indexer as the vLLM and sglang
// pages' workloads state them: key t of row i scores
//     s_t = sum_h w[i][h] * relu(scale * (q[i][h] . k_t) + b_i)
// over 64 heads of dimension 128 (bf16 q and k, fp32 accumulation and
// epilogue; b_i an optional per-row logit shift).
//
// Per 128-key tile the head logits are one MMA of M = 128 keys, N = 64
// heads per row, K = 128: A is the key tile, B the rows' queries, both
// K-major in shared memory with the 128-byte swizzle, staged by TMA.  An
// aligned block of four consecutive rows that read the same key window (the
// rows of a causal prefill chunk) is one group: its tiles take N = 256, so
// each key tile is loaded once for four rows.  The accumulator sits in tensor
// memory, one lane per key and one column per (row, head), so each epilogue
// thread owns one key and reduces a row's 64 heads alone, in a fixed order.
// Work is split evenly by tiles: the tiles of all groups, in row order, are
// cut into one contiguous range per CTA.
//
// Warp roles: warp 0 issues TMA loads (a ring of key tiles and a
// double-buffered query block), warp 1 owns the tensor memory and issues the
// MMAs, the other warps drain the accumulators (two of them, so the next
// tile's MMAs overlap this tile's epilogue) and write the scores.  Every
// wait is a bounded mbarrier wait.
//
// Two instances: IxCfg<1> never groups rows (a 4-stage ring, 16 KB query
// buffers, 4 epilogue warps: the shape of decode, where no two rows share
// keys and the key stream is the whole cost), IxCfg<4> groups them (a
// 3-stage ring, 64 KB query buffers, 8 epilogue warps, two per lane quarter,
// each taking every other row of a group).  Both are correct for any input;
// the host picks by how often the key buffer is shared.

constexpr int kIxHeads = 64;
constexpr int kIxDim = 128;
constexpr int kIxTile = 128;                                    // keys per tile (MMA M)
constexpr int kIxGroup = 4;                                     // most rows sharing a key tile
constexpr uint32_t kIxTileBytes = kIxTile * kIxDim * 2;         // 32 KB
constexpr uint32_t kIxHalfBytes = kIxTileBytes / 2;             // 64 dims of a tile: 16 KB

// Instruction descriptor of tcgen05.mma.kind::f16: f32 accumulator (bits
// 4-5 = 1), bf16 A and B (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 =
// 0), N / 8 in bits 17-22, M / 16 in bits 24-28.
__host__ __device__ constexpr uint32_t ix_idesc(uint32_t n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((uint32_t)(kIxTile >> 4) << 24);
}

template <int STAGES>
struct IxCtrl {
    uint64_t full[STAGES], empty[STAGES];
    uint64_t qfull[2], qempty[2];
    uint64_t afull[2], aempty[2];
    uint64_t scan64[32];
    uint32_t tmem;
    uint32_t first_row, first_tile;
    uint32_t edge[2];   // tile indices (in row order) that open this CTA's range and the next
};
template <int G>
struct IxCfg {
    static constexpr int kStages = G == 1 ? 4 : 3;              // key tiles in flight
    static constexpr int kEpiWarps = G == 1 ? 4 : 8;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    static constexpr uint32_t kQRows = G * kIxHeads;             // query rows per load
    static constexpr uint32_t kQBytes = kQRows * kIxDim * 2;     // 16 or 64 KB
    static constexpr uint32_t kQHalfBytes = kQBytes / 2;
    static constexpr uint32_t kAccCols = G * kIxHeads;           // columns per accumulator
    static constexpr uint32_t kTmemCols = 2 * kAccCols;          // 128 or 512
    // What a work unit's query load costs, in tiles: the split of the batch
    // weighs each unit as its tiles plus this, so CTAs that draw many short
    // units (the first rows of a causal chunk) draw fewer tiles.
    static constexpr uint32_t kUnitCost = G == 1 ? 1 : 4;
    // Dynamic shared memory: [ring: kStages x 32 KB][query: 2 x kQBytes]
    // [IxCtrl], from a 1024-byte aligned base (the 128-byte swizzle repeats
    // every 1 KB).
    static constexpr uint32_t kSmemBytes = kStages * kIxTileBytes + 2 * kQBytes + sizeof(IxCtrl<kStages>) + 1024;
};

struct IxParams {
    const float *w;                  // [B, 64]
    const float *bias;               // [B] or null
    const int32_t *key_starts;
    const int32_t *lengths;
    const int32_t *score_starts;
    float *scores;
    int64_t n_keys, n_scores;
    int32_t B;
    float scale;
};

// ---- PTX wrappers ---------------------------------------------------------- //
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int32_t x, int32_t y, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1 (bit 46).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Arrives on `bar` once every MMA this thread issued before it has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// 32 consecutive columns of this warp's 32 lanes: v[c] = column c of lane
// (warp's lane base + lane id).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
                 "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                   "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                   "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
                   "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---- rows and the walk over a CTA's tiles ----------------------------------- //
struct IxRow {
    int r;              // the group's first row
    uint32_t t;         // tile within the group
    uint32_t nt;        // tiles of the group
    uint32_t gsize;     // rows in the group (1 or kIxGroup)
    int32_t ks;         // the group's key window start
    int32_t L[kIxGroup], ss[kIxGroup];   // each member's valid length and score start
};

// Row r's own checks (topk_ragged's, on the key and the score window): its
// valid length (0 when rejected) and its status bit.
__device__ __forceinline__ int32_t ix_check(const IxParams &p, int r, int64_t &k0, int64_t &s0, uint32_t &bad)
{
    int64_t len = p.lengths[r];
    if (len < 0) len = 0;
    k0 = p.key_starts[r];
    s0 = p.score_starts[r];
    bad = 0;
    if (len >= (int64_t)TOPK_RAGGED_MAX_LEN)
        bad = TOPK_DEV_LEN_ENVELOPE;
    else if (k0 < 0 || k0 + len > p.n_keys || s0 < 0 || s0 + len > p.n_scores)
        bad = TOPK_DEV_BAD_WINDOW;
    return bad ? 0 : (int32_t)len;
}

// The work unit that starts at row r, and its tile count.  With G = 4, rows
// 4b..4b+3 form one group when all four exist, pass their checks and start
// at the same key; the group's later rows then have no tiles of their own.
// Every other row is a group of one.  `bad` is row r's own status bit.
template <int G>
__device__ __forceinline__ uint32_t ix_row(const IxParams &p, int r, IxRow &c, uint32_t &bad)
{
    int64_t k0, s0;
    const int32_t L0 = ix_check(p, r, k0, s0, bad);
    const int b0 = r & ~(kIxGroup - 1);
    bool grouped = G > 1 && b0 + kIxGroup <= p.B;
    int32_t Lm[kIxGroup];
    int64_t km[kIxGroup], sm[kIxGroup];
    if (grouped) {
#pragma unroll
        for (int m = 0; m < kIxGroup; ++m) {
            uint32_t bm;
            Lm[m] = ix_check(p, b0 + m, km[m], sm[m], bm);
            grouped = grouped && bm == 0 && km[m] == km[0];
        }
    }
    c.r = r;
    if (grouped) {
        c.gsize = kIxGroup;
        c.ks = (int32_t)km[0];
        int32_t Lmax = 0;
#pragma unroll
        for (int m = 0; m < kIxGroup; ++m) {
            c.L[m] = Lm[m];
            c.ss[m] = (int32_t)sm[m];
            Lmax = max(Lmax, Lm[m]);
        }
        c.nt = r == b0 ? (uint32_t)((Lmax + kIxTile - 1) / kIxTile) : 0u;
    } else {
        c.gsize = 1;
        c.ks = (int32_t)k0;
        c.L[0] = L0;
        c.ss[0] = (int32_t)s0;
#pragma unroll
        for (int m = 1; m < kIxGroup; ++m) {
            c.L[m] = 0;
            c.ss[m] = 0;
        }
        c.nt = (uint32_t)((L0 + kIxTile - 1) / kIxTile);
    }
    return c.nt;
}

// Next tile in row order (the caller knows one is left; the row bound is
// a guard that the tile count makes unreachable).
template <int G>
__device__ __forceinline__ void ix_next(const IxParams &p, IxRow &c)
{
    uint32_t bad;
    if (++c.t < c.nt) return;
    c.t = 0;
    do {
        if (c.r + 1 >= p.B) {
            c.gsize = 1;
            c.L[0] = 0;
            return;
        }
        ix_row<G>(p, c.r + 1, c, bad);
    } while (c.nt == 0);
}

template <int G>
__global__ void __launch_bounds__(IxCfg<G>::kThreads, 1)
    indexer_scores_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                          const IxParams p)
{
    using C = IxCfg<G>;
    constexpr int THREADS = C::kThreads;
    constexpr int kIxStages = C::kStages;
    constexpr int kIxEpiWarps = C::kEpiWarps;
    constexpr uint32_t kIxQBytes = C::kQBytes, kIxQHalfBytes = C::kQHalfBytes;
    constexpr uint32_t kIxAccCols = C::kAccCols, kIxTmemCols = C::kTmemCols;
    grid_dependency_enter();
    extern __shared__ unsigned char ix_smem_raw[];
    const uint32_t raw = smem_addr(ix_smem_raw);
    unsigned char *smem = ix_smem_raw + (((raw + 1023u) & ~1023u) - raw);
    unsigned char *ring = smem;
    unsigned char *qbuf = smem + kIxStages * kIxTileBytes;
    IxCtrl<kIxStages> &ctrl = *reinterpret_cast<IxCtrl<kIxStages> *>(qbuf + 2 * kIxQBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- this CTA's range of tiles ----------------------------------------- //
    // Per thread, a contiguous run of rows: its tiles and its weight (tiles
    // plus kUnitCost per work unit), then one 64-bit scan over the CTA.  CTA
    // b takes the tiles whose weighted positions fall in [b W / grid,
    // (b + 1) W / grid), a unit's cost counted before its first tile.
    {
        const int per = (p.B + THREADS - 1) / THREADS;
        const int lo = min(p.B, tid * per), hi = min(p.B, lo + per);
        uint64_t cnt = 0;   // weight << 32 | tiles
        uint32_t bad_any = 0;
        IxRow c;
        for (int r = lo; r < hi; ++r) {
            uint32_t bad;
            const uint32_t nt = ix_row<G>(p, r, c, bad);
            cnt += ((uint64_t)(nt ? nt + C::kUnitCost : 0u) << 32) | nt;
            bad_any |= bad;
        }
        if (bad_any && blockIdx.x == 0) atomicOr(&g_status, bad_any);
        uint64_t tot;
        const uint64_t incl = block_incl_scan64<THREADS>(cnt, ctrl.scan64, tot);
        const uint64_t excl = incl - cnt;
        const uint32_t W = (uint32_t)(tot >> 32);
        if (tid == 0) ctrl.edge[0] = ctrl.edge[1] = (uint32_t)tot;   // a position at W: past the last tile
        __syncthreads();
        for (int e = 0; e < 2; ++e) {
            const uint32_t pos = (uint32_t)((uint64_t)(blockIdx.x + e) * W / gridDim.x);
            if (pos < W && (uint32_t)(excl >> 32) <= pos && pos < (uint32_t)(incl >> 32)) {
                uint32_t pw = (uint32_t)(excl >> 32), pt = (uint32_t)excl;
                for (int r = lo; r < hi; ++r) {
                    uint32_t bad;
                    const uint32_t nt = ix_row<G>(p, r, c, bad);
                    const uint32_t wt = nt ? nt + C::kUnitCost : 0u;
                    if (pos < pw + wt) {
                        const uint32_t t = pos - pw < C::kUnitCost ? 0u : pos - pw - C::kUnitCost;
                        ctrl.edge[e] = pt + t;
                        if (e == 0) {
                            ctrl.first_row = (uint32_t)r;
                            ctrl.first_tile = t;
                        }
                        break;
                    }
                    pw += wt;
                    pt += nt;
                }
            }
        }
        if (tid == 0) {
            for (int s = 0; s < kIxStages; ++s) {
                mbar_init(&ctrl.full[s], 1);
                mbar_init(&ctrl.empty[s], 1);
            }
            for (int s = 0; s < 2; ++s) {
                mbar_init(&ctrl.qfull[s], 1);
                mbar_init(&ctrl.qempty[s], 1);
                mbar_init(&ctrl.afull[s], 1);
                mbar_init(&ctrl.aempty[s], kIxEpiWarps * 32);
            }
            mbar_init_fence();
        }
        __syncthreads();
    }
    const uint32_t n = ctrl.edge[1] - ctrl.edge[0];
    if (n == 0) return;   // uniform: nothing allocated yet
    IxRow start;
    {
        uint32_t bad;
        ix_row<G>(p, (int)ctrl.first_row, start, bad);
        start.t = ctrl.first_tile;
    }

    if (warp == 1) tmem_alloc(&ctrl.tmem, kIxTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl.tmem;

    if (warp == 0) {
        // ---- producer: query per row change, key tiles through the ring ---- //
        if (lane == 0) {
            IxRow c = start;
            int cur = -1;
            uint32_t qn = 0, stage = 0, sph = 0;
            for (uint32_t i = 0; i < n; ++i) {
                if (c.r != cur) {
                    const uint32_t qi = qn & 1u;
                    mbar_wait_bounded(&ctrl.qempty[qi], ((qn >> 1) & 1u) ^ 1u);
                    mbar_arrive_expect_tx(&ctrl.qfull[qi], kIxQBytes);
                    unsigned char *qd = qbuf + qi * kIxQBytes;
                    tma_load_2d(qd, &tmap_q, 0, c.r * kIxHeads, &ctrl.qfull[qi]);   // rows r..r+G-1
                    tma_load_2d(qd + kIxQHalfBytes, &tmap_q, 64, c.r * kIxHeads, &ctrl.qfull[qi]);
                    ++qn;
                    cur = c.r;
                }
                mbar_wait_bounded(&ctrl.empty[stage], sph ^ 1u);
                mbar_arrive_expect_tx(&ctrl.full[stage], kIxTileBytes);
                unsigned char *kd = ring + stage * kIxTileBytes;
                const int32_t y = c.ks + (int32_t)(c.t * kIxTile);
                tma_load_2d(kd, &tmap_k, 0, y, &ctrl.full[stage]);
                tma_load_2d(kd + kIxHalfBytes, &tmap_k, 64, y, &ctrl.full[stage]);
                if (++stage == kIxStages) {
                    stage = 0;
                    sph ^= 1u;
                }
                if (i + 1 < n) ix_next<G>(p, c);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer ---------------------------------------------------- //
        if (lane == 0) {
            IxRow c = start;
            int cur = -1;
            uint32_t qn = 0, qi = 0, stage = 0, sph = 0;
            for (uint32_t i = 0; i < n; ++i) {
                if (c.r != cur) {
                    if (cur >= 0) tc_commit(&ctrl.qempty[qi]);   // the last row's query, once its MMAs finish
                    qi = qn & 1u;
                    mbar_wait_bounded(&ctrl.qfull[qi], (qn >> 1) & 1u);
                    ++qn;
                    cur = c.r;
                }
                const uint32_t a = i & 1u;
                mbar_wait_bounded(&ctrl.aempty[a], ((i >> 1) & 1u) ^ 1u);
                mbar_wait_bounded(&ctrl.full[stage], sph);
                tc_fence_after();
                const uint32_t abase = smem_addr(ring + stage * kIxTileBytes);
                const uint32_t bbase = smem_addr(qbuf + qi * kIxQBytes);
                const uint32_t idesc = ix_idesc(c.gsize * (uint32_t)kIxHeads);   // N = 64 per row
#pragma unroll
                for (int kk = 0; kk < kIxDim / 16; ++kk) {
                    // 16 dims per MMA: 32 bytes into the 128-byte swizzle row,
                    // the second 64 dims in the second half.
                    const uint32_t off_a = (uint32_t)(kk >> 2) * kIxHalfBytes + (uint32_t)(kk & 3) * 32u;
                    const uint32_t off_b = (uint32_t)(kk >> 2) * kIxQHalfBytes + (uint32_t)(kk & 3) * 32u;
                    tc_mma(tmem + a * kIxAccCols, sw128_desc(abase + off_a), sw128_desc(bbase + off_b), idesc,
                           kk > 0 ? 1u : 0u);
                }
                tc_commit(&ctrl.empty[stage]);
                tc_commit(&ctrl.afull[a]);
                if (++stage == kIxStages) {
                    stage = 0;
                    sph ^= 1u;
                }
                if (i + 1 < n) ix_next<G>(p, c);
            }
        }
        __syncwarp();
    } else {
        // ---- epilogue: one key per thread, every other row of the group -- //
        const uint32_t quarter = (uint32_t)warp & 3u;   // the TMEM lanes this warp may read
        const uint32_t m0 = (uint32_t)(warp - 2) >> 2;  // 0 or 1: the group rows m0, m0 + 2
        const uint32_t key_in_tile = quarter * 32u + (uint32_t)lane;
        IxRow c = start;
        for (uint32_t i = 0; i < n; ++i) {
            const uint32_t a = i & 1u;
            mbar_wait_bounded(&ctrl.afull[a], (i >> 1) & 1u);
            tc_fence_after();
            const int32_t j = (int32_t)(c.t * kIxTile + key_in_tile);
            bool released = false;
            for (uint32_t m = m0; m < c.gsize; m += 2) {   // warp-uniform
                uint32_t v0[32], v1[32];
                const uint32_t taddr = tmem + ((quarter * 32u) << 16) + a * kIxAccCols + m * (uint32_t)kIxHeads;
                tmem_ld32(taddr, v0);
                tmem_ld32(taddr + 32u, v1);
                tmem_wait_ld();
                if (m + 2 >= c.gsize) {
                    // This warp's last read of the accumulator is in registers:
                    // release it before the arithmetic, so the MMAs of the
                    // tile after next can start.
                    tc_fence_before();
                    mbar_arrive(&ctrl.aempty[a]);
                    released = true;
                }
                if (j < c.L[m]) {
                    const int row = c.r + (int)m;
                    const float b = p.bias ? __ldg(p.bias + row) : 0.0f;
                    const float4 *wr = reinterpret_cast<const float4 *>(p.w + (int64_t)row * kIxHeads);
                    float s = 0.0f;
#pragma unroll
                    for (int h4 = 0; h4 < kIxHeads / 4; ++h4) {
                        const float4 ww = __ldg(wr + h4);
                        const uint32_t *v = h4 < 8 ? v0 + 4 * h4 : v1 + 4 * (h4 - 8);
                        s = fmaf(ww.x, fmaxf(fmaf(__uint_as_float(v[0]), p.scale, b), 0.0f), s);
                        s = fmaf(ww.y, fmaxf(fmaf(__uint_as_float(v[1]), p.scale, b), 0.0f), s);
                        s = fmaf(ww.z, fmaxf(fmaf(__uint_as_float(v[2]), p.scale, b), 0.0f), s);
                        s = fmaf(ww.w, fmaxf(fmaf(__uint_as_float(v[3]), p.scale, b), 0.0f), s);
                    }
                    p.scores[(int64_t)c.ss[m] + j] = s;
                }
            }
            if (!released) {   // a warp with no row of this group
                tc_fence_before();
                mbar_arrive(&ctrl.aempty[a]);
            }
            if (i + 1 < n) ix_next<G>(p, c);
        }
    }

    // Every MMA has completed (the epilogue consumed the last accumulator)
    // and every tensor-memory read has finished: give the columns back.
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kIxTmemCols);
    }
}
