// plan.h -- launch planning of the top-k kernels: pure host arithmetic over
// the call's (n_scores, B, k) and a description of the device, with no CUDA
// call, so that it can be checked on a machine without a GPU.
//
// The shared-memory layout of a CTA of either top-k kernel is
//
//   [ control block | histogram(s) | candidate list | staged keys ]
//   0               sizeof(ctrl)   off_win          off_keys      smem
//
// where the candidate list holds win_cap 8-byte composites and the staged
// keys stage_cap 4-byte keys, read and written as 16-byte vectors and by
// 16-byte bulk copies; off_keys is therefore kept a multiple of 128 bytes
// whatever win_cap is (k <= 2 gives a list of a single 8-byte slot).
#ifndef TOPK_PLAN_H
#define TOPK_PLAN_H

#include <stdint.h>

namespace topk_plan {

constexpr int kBins = 2048;                           // 11-bit digits
constexpr int kShortQuads = 4;                        // quads per thread, short-row path
constexpr int kShortScores = 4 * kShortQuads * 256;   // scores the one-CTA short path holds
constexpr int kRowCtasPerSm = 5;                      // the row kernel's launch bound

// Per-CTA control block of the one-CTA-per-row kernel.
struct alignas(16) Ctrl {
    uint32_t sel_digit;  // result of the last threshold search
    uint32_t sel_gt;     //   entries above the chosen bin (within the prefix)
    uint32_t sel_cnt;    //   entries in the chosen bin
    uint32_t sel_done;   //   1: the k-th key is +0.0 (plateau shortcut)
    uint32_t zeros;      // count of exact +0.0 scores
    uint32_t win_count;  // winner slots handed out
    uint32_t kmax;       // the largest order key
    uint32_t wmin;       // the smallest winner key
    uint32_t warp_zeros[32];
    uint32_t warp_ties[32];
    uint32_t scan[36];
    uint64_t scan64[32];
    // Short-row path: per-warp partials (non-zero count, smallest and
    // largest non-zero key) and the bucket statistics.
    uint32_t part_p[32], part_min[32], part_max[32];
    uint32_t sq;         // the largest bucket among those that are output
    uint32_t npart;      // entries in those buckets
};

// Per-CTA control block of the cluster kernel.
struct alignas(16) CCtrl {
    uint64_t bar[8];       // completion of each 32 KB bulk copy of the staged slice
    uint32_t zeros;        // this CTA's count of exact +0.0 keys
    uint32_t win_local;    // entries in this CTA's candidate list
    uint32_t wmin;         // smallest candidate key in this CTA's list
    uint32_t wmax;         // largest candidate key in this CTA's list
    uint32_t sel[4];       // threshold search result: digit, above, in bin
    uint32_t tot[4];       // group totals: +0.0 count
    uint32_t warp_zeros[32];
    uint32_t warp_ties[32];
    uint32_t scan[36];
    uint64_t scan64[32];
    // Sampled path: the sample's largest key, this CTA's candidate-list
    // overflow, the cluster's fallback flag (set remotely by any CTA whose
    // row group falls back), the largest fine bin of the group, the range
    // of this CTA's share of the group's candidates in its buffer, and the
    // sample's smallest positive key.
    uint32_t smax, overflow, cl_fb, maxbin;
    uint32_t loc_begin, loc_end, gz_before, smin;
    // Counters of the group's CTAs (entry g from the group's CTA g, written
    // into every CTA of the group before the cluster barrier).
    uint32_t gcnt[16];     // candidate-list lengths
    uint32_t gover[16];    // list overflow flags
    uint32_t gzero[16];    // +0.0 counts
    uint32_t gpos[17];     // first output place of each CTA's share (sampled path)
};

// Kernel variants: the one-CTA-per-row kernel and the cluster kernel at 512
// (two CTAs per SM) and 1024 threads (one CTA per SM).
enum { kRowKernel = 0, kCluster512 = 1, kCluster1024 = 2, kVariants = 3 };
constexpr int kVariantThreads[kVariants] = {256, 512, 1024};

// What the planner knows of a device.
struct DeviceShape {
    int sm_count;
    int max_smem;      // opt-in dynamic shared memory per block
    int smem_per_sm;   // shared memory per multiprocessor
    // max_clusters[variant][C]: co-resident clusters of C CTAs, each CTA with
    // the variant's budget (0 = not launchable)
    int max_clusters[kVariants][17];
};

struct Plan {
    int variant;
    int cluster;     // CTAs per cluster (1: no cluster)
    int stage_cap;   // scores per CTA staged in shared memory (multiple of 128)
    int win_cap;     // candidate slots (power of two)
    int off_win;     // byte offset of the candidate list
    int off_keys;    // byte offset of the staged keys (multiple of 128)
    int smem;        // dynamic shared memory per CTA
    int grid;        // CTAs launched
};

inline int next_pow2(int x)
{
    int n = 1;
    while (n < x) n <<= 1;
    return n;
}

inline int header_bytes(bool cluster)
{
    return cluster ? (int)sizeof(CCtrl) + 2 * kBins * 4 : (int)sizeof(Ctrl) + kBins * 4;
}

// Candidate slots: the one-CTA kernel keeps the winners (fewer than k); the
// cluster kernel keeps up to twice k candidates per CTA.
inline int list_cap(bool cluster, int k)
{
    // The cluster kernel's list also holds the 4096-bin histogram of the
    // row's sample before the candidates are appended: 2048 slots at least.
    return cluster ? (2 * next_pow2(k) > 2048 ? 2 * next_pow2(k) : 2048) : next_pow2(k - 1 > 1 ? k - 1 : 1);
}

// Dynamic shared memory a CTA of the variant may use: all an SM has for the
// 1024-thread cluster kernel, half of it for the 512-thread one (two CTAs
// per SM, each leaving the runtime's 1 KB reserve).
inline int variant_budget(const DeviceShape &dev, int v)
{
    return v == kCluster1024 ? dev.max_smem : dev.smem_per_sm / 2 - 1024;
}

inline int stage_cap_for(int smem_budget, int off_keys)
{
    return ((smem_budget - off_keys) / 4) & ~127;
}

inline int keys_offset(int off_win, int win_cap)
{
    return (off_win + win_cap * 8 + 127) & ~127;
}

// Launch shape from the host arguments alone (row lengths live on the
// device and are never read here).
//   * B >= 4 x SMs, or short rows on average: one 256-thread CTA per row,
//     several CTAs per SM.
//   * otherwise one resident wave of G clusters of CS CTAs, either
//     1024-thread CTAs with all of an SM's shared memory or 512-thread CTAs
//     two to an SM; the clusters share out the rows by length and each
//     cluster deals its CTAs to its rows so that the largest slice is as
//     small as possible.  Of the shapes that give every row a CTA, the
//     planner takes the one whose typical row gets the most staging
//     capacity, min(CS, G x CS / B) x scores staged per CTA, and on a tie the
//     one with more CTAs.  A variant whose budget cannot hold the sort's
//     second buffer (2 x the candidate list) is not considered.
// Each CTA stages what shared memory allows and re-reads the rest of its
// slice from L2.
inline Plan make_plan(int64_t n_scores, int32_t B, int32_t k, const DeviceShape &dev)
{
    Plan pl{};
    const int sms = dev.sm_count;
    const int wcap_cluster = list_cap(true, k);
    const int off_keys_cluster = keys_offset(header_bytes(true), wcap_cluster);
    int vi = kRowKernel, cluster = 1, smem_budget = 0, grid = B;
    // Short rows on average (the buffer holds at most kShortScores scores per
    // row) go to the one-CTA-per-row kernel, whose short path ranks such a
    // row in registers; clusters pay off for longer rows.
    const bool short_rows = n_scores <= (int64_t)B * kShortScores;
    if (B < 4 * sms && !short_rows) {
        double best = 0.0;
        for (int v = kCluster1024; v >= kCluster512; --v) {
            const int budget = variant_budget(dev, v);
            const int cap = stage_cap_for(budget, off_keys_cluster);
            // The staging area doubles as the sort's second buffer.
            if (cap < 2 * wcap_cluster) continue;
            for (int cs = 2; cs <= 16; cs *= 2) {
                int g = dev.max_clusters[v][cs];
                if (v == kCluster512 && g > 2 * sms / cs) g = 2 * sms / cs;
                if (g <= 0 || (int64_t)g * cs < B) continue;
                const double rows_per = (double)g * cs / B;
                const double share = (rows_per < cs ? rows_per : (double)cs) * cap;
                if (share > best * 1.0001 || (share > best * 0.9999 && g * cs > grid)) {
                    best = share;
                    vi = v;
                    cluster = cs;
                    smem_budget = budget;
                    grid = g * cs;
                }
            }
        }
    }
    const bool is_cluster = vi != kRowKernel;
    pl.variant = vi;
    pl.cluster = cluster;
    pl.win_cap = list_cap(is_cluster, k);
    pl.off_win = header_bytes(is_cluster);
    pl.off_keys = keys_offset(pl.off_win, pl.win_cap);
    int stage_cap = is_cluster ? stage_cap_for(smem_budget, pl.off_keys) : 4096 + 256;
    // The row kernel's staging area also doubles as the sort's second buffer.
    if (stage_cap < 2 * pl.win_cap) stage_cap = 2 * pl.win_cap;
    pl.stage_cap = stage_cap;
    pl.smem = pl.off_keys + stage_cap * 4;
    pl.grid = grid;
    return pl;
}

}  // namespace topk_plan

#endif  // TOPK_PLAN_H
