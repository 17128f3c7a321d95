/*
 * oracle.c -- plain, slow CPU oracle for deterministic exact ragged top-k.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline / reference arm use it.  It shares no code, header, table or
 * constant with the CUDA library; it is written directly from the definition
 * of the selection the source pages give.
 *
 * What it computes (per row i):
 *   window      scores[row_starts[i] .. row_starts[i] + L_i), L_i = lengths[i]
 *               (negative lengths read as 0);
 *   order       the bitwise total order on fp32 bit patterns: every pattern u
 *               maps to an unsigned 32-bit order key, larger key ranks first,
 *               and among bitwise-equal scores the smaller row-local index
 *               ranks first; NaNs take their place in that bit order
 *               instead of all ranking first as in torch.topk (sglang PR
 *               #31115 "Add opt-in deterministic CuTe-DSL DSA top-k
 *               backend", PR summary and the hardening commit message);
 *   selection   the first n = min(k, L_i) entries of that order, which is the
 *               smallest-index subset of the tie set at the k-th boundary
 *               (same page, PR summary; Modifications);
 *   output      out_idx[i, p] = row-local index (offset_mode 0) or
 *               row_starts[i] + index (offset_mode 1) for p < n, -1 for
 *               p >= n (rows packed from the front and filled with -1, same
 *               page, Modifications;
 *               the -1 padding when length < k also appears in the blog post
 *               "Non-deterministic Qwen3.8-Flash-Next: we found the faulty
 *               vLLM kernel and fixed it", section "The price of the fix");
 *               out_val[i, p] = the selected entry's original fp32 bits, and
 *               -inf bits (0xFF800000) in the padding (the pages name no pad
 *               value; -inf is this library's reading).
 *   envelope    a length >= 2^24 breaks the 24-bit inverted-index composite
 *               the pages' kernel relies on (the index field wraps; same
 *               page, hardening commit); such a row is written as all -1 and
 *               flagged (bit 1).  A window not inside [0, n_scores) is written
 *               as all -1 and flagged (bit 2): the flat-buffer reading of the
 *               same commit's clamping of windows against trusted metadata.
 *   exclusion   with offset_mode bit 2 set, the scores at or below -inf in the
 *               total order (-inf and every negative NaN) are left out
 *               before the selection: the row holds the first min(k, m) of
 *               the m remaining entries, then -1.  This reads the sglang
 *               page's torch-compatible backend (Modifications), which
 *               leaves -inf scores out; the negative NaNs, which rank below
 *               -inf, go with them, so the excluded entries are exactly a
 *               tail of the order.
 *
 * Method: per row, build (order key, index) pairs and sort them with qsort
 * under an explicit comparator.  No blocking, no radix, no fusion.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAX_K 4096
#define ORACLE_MAX_LEN ((int64_t)1 << 24)
#define ORACLE_FLAG_LEN_ENVELOPE 1u
#define ORACLE_FLAG_BAD_WINDOW 2u
/* offset_mode bits: indices offset by the row start; -inf excluded. */
#define ORACLE_OFFSET_ROW_START 1
#define ORACLE_EXCLUDE_NEG_INF 2

/* Order key of one fp32 bit pattern.  For a non-negative float (sign bit
 * clear) setting the sign bit moves it above every negative pattern while
 * keeping magnitude order; for a negative float, inverting all bits reverses
 * magnitude order (a larger magnitude is a smaller number) and clears the top
 * bit.  This is the total order on bit patterns of the hardening commit: -NaN
 * below -inf, -0.0 just below +0.0, +NaN above +inf, NaN payloads ordered by
 * their bits. */
uint32_t oracle_order_key(uint32_t bits)
{
    if (bits & 0x80000000u)
        return ~bits;
    return bits | 0x80000000u;
}

void oracle_order_key_batch(const uint32_t *in, uint32_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_order_key(in[i]);
}

typedef struct {
    uint32_t key;
    int32_t idx;
} oracle_pair;

/* Canonical order: larger key first; on equal keys, smaller index first. */
static int oracle_cmp(const void *pa, const void *pb)
{
    const oracle_pair *a = (const oracle_pair *)pa;
    const oracle_pair *b = (const oracle_pair *)pb;
    if (a->key != b->key)
        return a->key > b->key ? -1 : 1;
    if (a->idx != b->idx)
        return a->idx < b->idx ? -1 : 1;
    return 0;
}

typedef struct {
    const float *scores;
    int64_t n_scores;
    const int32_t *row_starts;
    const int32_t *lengths;
    int32_t B, k, offset_mode;
    int32_t *out_idx;
    float *out_val;
    uint32_t *row_flags;
    int thread_id, n_threads;
    int failed;
} oracle_job;

static void oracle_pad_row(const oracle_job *job, int64_t row, int32_t from)
{
    const uint32_t neg_inf_bits = 0xFF800000u;
    for (int32_t p = from; p < job->k; ++p) {
        job->out_idx[row * job->k + p] = -1;
        if (job->out_val)
            memcpy(&job->out_val[row * job->k + p], &neg_inf_bits, 4);
    }
}

static void *oracle_worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    oracle_pair *pairs = NULL;
    int64_t cap = 0;
    /* Rows are dealt round-robin so that ragged lengths spread evenly. */
    for (int64_t row = job->thread_id; row < job->B; row += job->n_threads) {
        int64_t start = job->row_starts[row];
        int64_t len = job->lengths[row];
        uint32_t flags = 0;
        if (len < 0)
            len = 0;
        if (len >= ORACLE_MAX_LEN)
            flags |= ORACLE_FLAG_LEN_ENVELOPE;
        else if (start < 0 || start + len > job->n_scores)
            flags |= ORACLE_FLAG_BAD_WINDOW;
        if (job->row_flags)
            job->row_flags[row] = flags;
        if (flags) {
            oracle_pad_row(job, row, 0);
            continue;
        }
        if (len > cap) {
            free(pairs);
            cap = len;
            pairs = (oracle_pair *)malloc((size_t)cap * sizeof(oracle_pair));
            if (!pairs) {
                job->failed = 1;
                return NULL;
            }
        }
        /* With the exclusion flag the scores at or below -inf in the total
         * order (-inf and every negative NaN) are not candidates at all. */
        const int exclude = (job->offset_mode & ORACLE_EXCLUDE_NEG_INF) != 0;
        const uint32_t neg_inf_key = oracle_order_key(0xFF800000u);
        int64_t m = 0;
        for (int64_t j = 0; j < len; ++j) {
            uint32_t bits;
            memcpy(&bits, &job->scores[start + j], 4);
            const uint32_t key = oracle_order_key(bits);
            if (exclude && key <= neg_inf_key)
                continue;
            pairs[m].key = key;
            pairs[m].idx = (int32_t)j;
            ++m;
        }
        qsort(pairs, (size_t)m, sizeof(oracle_pair), oracle_cmp);
        int32_t n = m < job->k ? (int32_t)m : job->k;
        for (int32_t p = 0; p < n; ++p) {
            int32_t j = pairs[p].idx;
            job->out_idx[row * job->k + p] =
                (job->offset_mode & ORACLE_OFFSET_ROW_START) ? (int32_t)(start + j) : j;
            if (job->out_val)
                job->out_val[row * job->k + p] = job->scores[start + j];
        }
        oracle_pad_row(job, row, n);
    }
    free(pairs);
    return NULL;
}

/* Returns 0 on success, -1 on an argument the selection does not define
 * (k outside [1, 4096], B < 0, offset_mode other than a combination of
 * ORACLE_OFFSET_ROW_START and ORACLE_EXCLUDE_NEG_INF, a null buffer),
 * -2 if a worker could not allocate its pair buffer.  row_flags (nullable)
 * receives the per-row envelope/window flags described above. */
int oracle_topk_ragged(const float *scores, int64_t n_scores,
                       const int32_t *row_starts, const int32_t *lengths,
                       int32_t B, int32_t k, int32_t offset_mode,
                       int32_t *out_idx, float *out_val, uint32_t *row_flags,
                       int n_threads)
{
    if (k < 1 || k > ORACLE_MAX_K || B < 0 || (offset_mode & ~3) != 0)
        return -1;
    if (B == 0)
        return 0;
    if (!row_starts || !lengths || !out_idx || (!scores && n_scores > 0) || n_scores < 0)
        return -1;
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > B)
        n_threads = B;
    oracle_job *jobs = (oracle_job *)calloc((size_t)n_threads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    for (int t = 0; t < n_threads; ++t) {
        oracle_job j = {scores, n_scores, row_starts, lengths, B, k, offset_mode,
                        out_idx, out_val, row_flags, t, n_threads, 0};
        jobs[t] = j;
    }
    int started = 0;
    for (int t = 1; t < n_threads; ++t) {
        if (pthread_create(&tids[t], NULL, oracle_worker, &jobs[t]) != 0)
            break;
        started = t;
    }
    /* Rows of threads that could not be started run on this thread. */
    for (int t = started + 1; t < n_threads; ++t)
        oracle_worker(&jobs[t]);
    oracle_worker(&jobs[0]);
    int failed = jobs[0].failed;
    for (int t = 1; t <= started; ++t) {
        pthread_join(tids[t], NULL);
        failed |= jobs[t].failed;
    }
    for (int t = started + 1; t < n_threads; ++t)
        failed |= jobs[t].failed;
    free(jobs);
    free(tids);
    return failed ? -2 : 0;
}
