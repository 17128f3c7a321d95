/*
 * topk_ragged.h -- C ABI of the deterministic exact ragged top-k library.
 *
 * The operation is the index-selection step of a DSA/QSA sparse-attention
 * lightning indexer: for each query row pick the k (default 2048, at most
 * 4096) highest-scoring key positions.  Its definition follows sglang PR
 * #31115 "Add opt-in deterministic CuTe-DSL DSA top-k backend" (PR summary;
 * Modifications; the hardening commit):
 *
 *   - canonical order: score descending, ascending index on bitwise-equal
 *     scores, so at the k-th boundary the smallest-index subset of the tie set
 *     is kept and no candidate is ever dropped;
 *   - the order on scores is the bitwise total order of fp32 patterns: each
 *     pattern u maps to the unsigned key (u & 0x80000000) ? ~u : u | 0x80000000
 *     and a larger key ranks first, so -NaN < -inf < ... < -0.0 < +0.0 < ...
 *     < +inf < +NaN, with NaN payloads ordered by their bits (not torch.topk's
 *     NaN-maximal order);
 *   - output rows are front-packed: the min(k, L_i) selected indices in
 *     canonical order, then -1.
 *
 * Around the selection the library offers its neighbours in the indexer
 * pipeline: the selection written as KV-cache slots through a page table
 * (topk_ragged_paged), per-row tie / plateau statistics at the k-th boundary
 * (topk_ragged_stats), and the indexer scores themselves on the tcgen05
 * tensor cores, alone or chained with the selection (topk_ragged_indexer_scores,
 * topk_ragged_indexer).
 *
 * Every call is stream-ordered and asynchronous, allocates nothing, and may be
 * captured into a CUDA graph once topk_ragged_init() has run for the device.
 * Results are bitwise identical from run to run and independent of which
 * other rows share the batch.
 */
#ifndef TOPK_RAGGED_H
#define TOPK_RAGGED_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TOPK_RAGGED_ABI_VERSION 4
#define TOPK_RAGGED_MAX_K 4096
/* Row lengths must stay below 2^24, the envelope of the 24-bit index field. */
#define TOPK_RAGGED_MAX_LEN (1 << 24)

/* Synchronous return codes. */
typedef enum {
    TOPK_OK = 0,
    TOPK_ERR_INVALID_ARG = 1,        /* an argument outside the contract below  */
    TOPK_ERR_NOT_INITIALIZED = 2,    /* called under stream capture before init */
    TOPK_ERR_UNSUPPORTED_DEVICE = 3, /* not a compute-capability 10.3 device    */
    TOPK_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed    */
    TOPK_ERR_SCRATCH_TOO_SMALL = 5   /* n_scores beyond the library's fixed
                                        score array (topk_ragged_indexer_static) */
} topk_status;

/* offset_mode: TOPK_OFFSET_ROW_LOCAL or TOPK_OFFSET_ROW_START, optionally
 * or-ed with TOPK_EXCLUDE_NEG_INF. */
enum {
    TOPK_OFFSET_ROW_LOCAL = 0, /* out_idx holds j, the index inside the row      */
    TOPK_OFFSET_ROW_START = 1, /* out_idx holds row_starts[i] + j (buffer index) */
    /* Leave out -inf and every negative NaN (the scores at or below -inf in
     * the order): the row holds the selection of its other entries, front-
     * packed, then -1.  The torch-compatible backend of sglang PR #31115
     * (Modifications) leaves -inf scores out; without this bit -inf ranks by
     * its key like any score. */
    TOPK_EXCLUDE_NEG_INF = 2
};

/* Bits of the device status word (data errors found by the kernel). */
enum {
    TOPK_DEV_LEN_ENVELOPE = 1u, /* a row had lengths[i] >= 2^24; it was written as all -1   */
    TOPK_DEV_BAD_WINDOW = 2u,   /* a row window left [0, n_scores); it was written as all -1 */
    TOPK_DEV_INTERNAL = 4u      /* an internal check failed or a bounded wait ran out; the   */
                                /* call's output rows are undefined                          */
};

/* Version of this ABI (TOPK_RAGGED_ABI_VERSION). */
int topk_ragged_abi_version(void);

/* Static description of a status code; never NULL. */
const char *topk_ragged_strerror(int status);

/*
 * Prepares `device` (0-based CUDA ordinal): checks that it is a
 * compute-capability 10.3 GPU, sets the kernels' shared-memory and cluster
 * attributes, and records the SM count used to size launches.  Idempotent and
 * thread-safe.  Must run outside stream capture; topk_ragged() calls it
 * itself on first use when the stream is not capturing.  The calling
 * thread's current device is the same on return as on entry.
 * Returns TOPK_OK, TOPK_ERR_UNSUPPORTED_DEVICE or TOPK_ERR_CUDA.
 */
int topk_ragged_init(int device);

/*
 * Exact top-k of every row of a flat ragged fp32 buffer (the
 * `topk_func(score, lengths, topk, row_starts)` contract of the page above,
 * with the 2-D score tensor replaced by one flat buffer and per-row windows).
 *
 * scores       device, fp32, n_scores entries, 4-byte aligned, read-only.
 * n_scores     number of entries in `scores`, 0 <= n_scores < 2^31.  Every
 *              row window must lie inside [0, n_scores); a row whose window
 *              does not is written as all -1 and TOPK_DEV_BAD_WINDOW is set.
 * row_starts   device, int32[B]: row i's window starts at scores[row_starts[i]].
 * lengths      device, int32[B]: L_i = lengths[i]; a negative length reads as 0;
 *              L_i >= 2^24 writes the row as all -1 and sets TOPK_DEV_LEN_ENVELOPE.
 *              Windows may overlap, be unaligned and come in any order.
 * B            number of rows, B >= 0; B == 0 returns TOPK_OK with no launch.
 * k            1 <= k <= 4096, and (int64)B * k < 2^31.
 * offset_mode  TOPK_OFFSET_ROW_LOCAL or TOPK_OFFSET_ROW_START, optionally
 *              or-ed with TOPK_EXCLUDE_NEG_INF.
 * out_idx      device, int32[B, k] row-major, written entirely: row i holds
 *              the min(k, L_i) selected indices in canonical order, then -1.
 * out_val      device, fp32[B, k] or NULL: the selected scores' original bit
 *              patterns (NaN payloads and the sign of zero survive), and -inf
 *              in the -1 slots.
 * stream       cudaStream_t to run on (NULL = legacy default stream).
 *
 * All buffers are owned by the caller and must stay valid until the stream
 * reaches the call.  Output buffers must not overlap the inputs.  The call
 * allocates no memory.  Returns TOPK_OK, TOPK_ERR_INVALID_ARG (nothing is
 * launched), TOPK_ERR_NOT_INITIALIZED, TOPK_ERR_UNSUPPORTED_DEVICE or
 * TOPK_ERR_CUDA.  Data errors are reported through
 * topk_ragged_device_status().
 */
int topk_ragged(const float *scores, int64_t n_scores, const int32_t *row_starts,
                const int32_t *lengths, int32_t B, int32_t k, int32_t offset_mode,
                int32_t *out_idx, float *out_val, void *stream);

/*
 * topk_ragged with every selected index written as a KV-cache slot through a
 * page table: the transform both engines on the pages run right after the
 * selection (vLLM PR #55872 calls FlashInfer's top_k_ragged_transform;
 * sglang PR #31115's Modifications note that its selection-only backends
 * leave out the fused page-table transforms).  Row i's selected in-row index
 * j is written as
 *     page_table[i * page_table_stride + j / page_size] * page_size
 *         + j % page_size,
 * in canonical order, then -1.
 *
 * flags              0 or TOPK_EXCLUDE_NEG_INF (a row-start offset has no
 *                    meaning here and is rejected).
 * page_table         device, int32: row i's pages start at
 *                    page_table + i * page_table_stride and must number at
 *                    least ceil(L_i / page_size); every slot must fit int32.
 * page_table_stride  >= 0 (0: all rows read one page table).
 * page_size          >= 1.
 * Everything else as for topk_ragged, with the same return codes.
 */
int topk_ragged_paged(const float *scores, int64_t n_scores, const int32_t *row_starts,
                      const int32_t *lengths, int32_t B, int32_t k, int32_t flags,
                      const int32_t *page_table, int64_t page_table_stride, int32_t page_size,
                      int32_t *out_idx, float *out_val, void *stream);

/*
 * Tie / plateau statistics of one row at its k-th boundary: the per-row
 * figures of the sglang page's score-statistics script (row_stats: plateau
 * fraction, the k-th score, its tie set, the count strictly above it,
 * straddle, zero_bound), taken on the selection's bitwise order.
 */
typedef struct {
    uint32_t len;            /* L_i after clamping (0 for a rejected row)           */
    uint32_t n_zero;         /* entries whose value is 0.0 (+0.0 or -0.0)          */
    uint32_t boundary_bits;  /* fp32 bits of the k-th entry in canonical order     */
    uint32_t tie;            /* entries bitwise equal to the boundary              */
    uint32_t above;          /* entries above the boundary in the order (L if L<=k)*/
    uint32_t flags;          /* TOPK_STAT_* bits                                   */
} topk_row_stats;

enum {
    TOPK_STAT_HAS_BOUNDARY = 1u, /* L_i > k; otherwise boundary_bits and tie are 0  */
    TOPK_STAT_STRADDLE = 2u,     /* tie > 1 and above + tie > k: the selection takes
                                    part of the tie set, by index                   */
    TOPK_STAT_ZERO_BOUND = 4u    /* the boundary score is 0.0 (either sign)         */
};

/*
 * Fills out[i] (device memory, B entries, caller-owned) with the statistics
 * of row i for this k.  Same inputs, window checks and status bits as
 * topk_ragged: a row outside [0, n_scores) or with L_i >= 2^24 is written
 * as all zero and sets its TOPK_DEV_* bit.  One launch, stream-ordered, no
 * allocation, capturable after topk_ragged_init.  Returns TOPK_OK,
 * TOPK_ERR_INVALID_ARG (k outside [1, 4096], B < 0, n_scores outside
 * [0, 2^31), NULL pointers with B > 0, scores not 4-byte aligned),
 * TOPK_ERR_NOT_INITIALIZED, TOPK_ERR_UNSUPPORTED_DEVICE or TOPK_ERR_CUDA.
 */
int topk_ragged_stats(const float *scores, int64_t n_scores, const int32_t *row_starts,
                      const int32_t *lengths, int32_t B, int32_t k, topk_row_stats *out,
                      void *stream);

/*
 * Lightning-indexer scores on the tensor cores (tcgen05 MMAs fed by TMA):
 * key t of row i scores
 *     s_t = sum over h < 64 of w[i][h] * relu(scale * (q[i][h] . k_t) + bias[i])
 * with 64 heads of dimension 128, the indexer of the vLLM and sglang pages'
 * decode and prefill workloads (bias is an optional per-row logit shift).
 * Products and sums run in fp32 on the tensor cores; the epilogue sums the
 * heads in index order with fused multiply-adds, so a call is deterministic.
 *
 * q             device, bf16 bit patterns, [B][64][128], 16-byte aligned.
 * w             device fp32 [B][64], 16-byte aligned.
 * bias          device fp32 [B], or NULL for 0.
 * keys          device, bf16 bit patterns, [n_keys][128], 16-byte aligned;
 *               1 <= n_keys <= 2^31 - 128.
 * key_starts, lengths, score_starts
 *               device int32 [B]: row i reads keys[key_starts[i] + j] and
 *               writes scores[score_starts[i] + j] for j < L_i (a negative
 *               length reads as 0).  Rows may share keys (a causal prefill
 *               chunk) and must not share score windows.
 * scores        device fp32 [n_scores], caller-owned; only the rows' score
 *               windows are written.
 * A row whose key or score window leaves its buffer, or with L_i >= 2^24,
 * writes nothing and sets its TOPK_DEV_* bit.  Inputs must be finite (a NaN
 * logit reads as 0 through the relu).  One launch, stream-ordered, no
 * allocation, capturable after topk_ragged_init.  Returns TOPK_OK,
 * TOPK_ERR_INVALID_ARG (B < 0, B * 64 >= 2^31, n_keys or n_scores out of
 * range, a non-finite scale, NULL or misaligned pointers),
 * TOPK_ERR_NOT_INITIALIZED, TOPK_ERR_UNSUPPORTED_DEVICE or TOPK_ERR_CUDA.
 */
int topk_ragged_indexer_scores(const uint16_t *q, const float *w, const float *bias, const uint16_t *keys,
                               int64_t n_keys, const int32_t *key_starts, const int32_t *lengths,
                               const int32_t *score_starts, int32_t B, float scale, float *scores,
                               int64_t n_scores, void *stream);

/*
 * The indexer scores into the caller's `scores` buffer, then topk_ragged over
 * them (row i's window: score_starts[i], L_i): two launches on `stream`.
 * Indices are row-local (j, the key's place in the row's key window);
 * flags is 0 or TOPK_EXCLUDE_NEG_INF.  Arguments and errors as for the two
 * calls.
 */
int topk_ragged_indexer(const uint16_t *q, const float *w, const float *bias, const uint16_t *keys,
                        int64_t n_keys, const int32_t *key_starts, const int32_t *lengths,
                        const int32_t *score_starts, int32_t B, float scale, float *scores, int64_t n_scores,
                        int32_t k, int32_t flags, int32_t *out_idx, float *out_val, void *stream);

/*
 * topk_ragged_indexer for callers that cannot allocate device memory.  The
 * chain's intermediate scores go to a score array that the library itself
 * holds, not to a caller buffer, so the caller provides only the inputs and
 * the outputs.  Callers that cannot allocate include code that runs inside
 * a framework which reserves the device memory for its own allocator or
 * cache up front (a plugin has no budget left to call cudaMalloc with, and
 * a call would fail or fragment the pool), and code on a latency-critical
 * path where cudaMalloc would synchronize the device or is not allowed at
 * all (cudaMalloc is refused while a stream is captured in the global mode).
 * The sources this library follows have no counterpart of this entry point;
 * it is an addition of this library.
 *
 * The array holds TOPK_RAGGED_STATIC_SCORES fp32 scores (32 MiB).  Every GPU
 * on which the library is loaded keeps it until the process exits.
 * score_starts and n_scores lay the rows' score windows out inside it as
 * they would inside a caller buffer: each window inside [0, n_scores), no
 * two rows sharing a window.  0 <= n_scores <= TOPK_RAGGED_STATIC_SCORES;
 * a larger n_scores returns TOPK_ERR_SCRATCH_TOO_SMALL and launches nothing.
 *
 * All calls on a device share the array, and each leaves its scores in it.
 * Nothing in it has to start at zero: the score kernel writes every entry of
 * a row's window before the selection reads it, and entries outside the
 * windows are never read.  Calls whose work overlaps on the GPU (two
 * streams, or two host threads, with nothing ordering them) race on the
 * array and can read each other's scores: order them on one stream or with
 * events.
 *
 * The first call on a device looks up the array's device address, with that
 * device current, and keeps it for the later calls.  Make that first call
 * outside stream capture: a first call under capture returns
 * TOPK_ERR_NOT_INITIALIZED and launches nothing.  Everything else -- the
 * arguments, the two launches on `stream`, the outputs, the device status
 * bits and the return codes -- is as for topk_ragged_indexer.  The call
 * allocates nothing.
 */
#define TOPK_RAGGED_STATIC_SCORES (1 << 23)
int topk_ragged_indexer_static(const uint16_t *q, const float *w, const float *bias, const uint16_t *keys,
                               int64_t n_keys, const int32_t *key_starts, const int32_t *lengths,
                               const int32_t *score_starts, int32_t B, float scale, int64_t n_scores,
                               int32_t k, int32_t flags, int32_t *out_idx, float *out_val, void *stream);

/*
 * Reads the current device's status word (an OR of TOPK_DEV_* bits from all
 * calls since the last read) into *host_out, then clears it.  Synchronizes
 * `stream`; not for use under stream capture.  Returns TOPK_OK,
 * TOPK_ERR_INVALID_ARG (host_out NULL) or TOPK_ERR_CUDA.
 */
int topk_ragged_device_status(uint32_t *host_out, void *stream);

/*
 * Diagnostic of the kernels' bounded waits (no counterpart on the pages: it
 * checks the library's own safety net).  Every wait in the kernels -- on an
 * mbarrier that a bulk copy or a tensor-core commit completes -- polls a
 * bounded number of times.  When the bound runs out the kernel sets
 * TOPK_DEV_INTERNAL in the status word, waits once more (again bounded) for
 * what it may still have in flight, and goes on, so the context stays usable;
 * the output rows of that call are then undefined.  This entry point launches
 * one CTA that makes such a wait, with `polls` polls per bound, on an
 * mbarrier that nothing completes: after it, topk_ragged_device_status reads
 * TOPK_DEV_INTERNAL instead of the call hanging.  Each poll may suspend the
 * thread for a short time the hardware chooses, so the probe takes about
 * `polls` microseconds at most.
 *
 * polls   1 .. 2^22 (the kernels' own bound).
 * stream  CUDA stream (cudaStream_t), or NULL.
 * Returns TOPK_OK, TOPK_ERR_INVALID_ARG (polls out of range), the init error
 * or TOPK_ERR_CUDA.
 */
int topk_ragged_wait_probe(uint32_t polls, void *stream);

/* How a call with these host arguments is launched on the current device. */
typedef struct {
    int32_t threads;        /* threads per CTA                                */
    int32_t cluster;        /* CTAs per row (a thread-block cluster)          */
    int32_t stage_cap;      /* scores per CTA held in shared memory           */
    int32_t smem_bytes;     /* dynamic shared memory per CTA                  */
    int32_t grid;           /* CTAs launched                                  */
    int32_t launches;       /* kernel launches per call (0 when B == 0)       */
} topk_launch_info;

/*
 * Fills *info for a call with (n_scores, B, k) on the current device without
 * launching anything.  Returns TOPK_OK, TOPK_ERR_INVALID_ARG or the init
 * error.
 */
int topk_ragged_launch_info(int64_t n_scores, int32_t B, int32_t k, topk_launch_info *info);

#ifdef __cplusplus
}
#endif

#endif /* TOPK_RAGGED_H */
