/*
 * topk_oracle.c -- plain, slow, obviously correct CPU definition of the
 * sparse-attention indexer's top-k + page-table transform.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this library.  The CUDA library never
 * links, includes or calls it, and it shares no code, header, table or
 * constant with the CUDA sources.
 *
 * What is computed (SGLang PR #26788 "[JIT Kernel] DeepSeek-V4 DSA indexer:
 * faster top-k + page-table transform (runtime k <= 2048)", sections
 * "Motivation" and "Feature"): for every row b of the score matrix, select
 * the k positions with the largest scores among the row's first seq_len[b]
 * entries, map each selected position idx through the row's page table
 *
 *     out = page_table[b][idx / page_size] * page_size + idx % page_size
 *
 * and pad the slots past min(k, seq_len) with -1.  The optional raw output
 * holds the selected positions before the transform, slot-aligned with out
 * (same PR, commit "Add an optional raw-index output to
 * topk_transform_512_v2").
 *
 * The selection is written as its plain definition: a full sort of the row.
 *   - Order: larger score first, compared as IEEE floats, so -0.0 == +0.0.
 *   - Ties: the pages leave the winner among equal scores open (the LiteTopk
 *     PR #32094, section "Notes", takes arrival order).  Here the smaller
 *     position wins, which makes the selected set unique.  The sort below
 *     compares (score, position) so the order is total and qsort's lack of
 *     stability cannot matter.
 *   - NaN is outside every workload; it is given a fixed place so that the
 *     result is still defined: a NaN with the sign bit clear ranks above
 *     +inf, a NaN with the sign bit set ranks below -inf.  Among positive
 *     NaNs the larger bit pattern ranks higher; among negative NaNs the larger
 *     bit pattern ranks lower.
 *   - -inf is an ordinary (lowest non-NaN) score and can be selected.
 *   - seq_len < 0 counts as 0 (SGLang PR #31123 "Harden top-k v1/v2 kernels
 *     against negative padded seq_lens", referenced from PR #26788); seq_len
 *     > max_seq_len is clamped to max_seq_len and reported in the flags.
 *   - The transform is evaluated in 32-bit two's-complement arithmetic
 *     (wrap-around), page_size is a power of two (PR #26788, "Feature").
 *
 * Rows are independent; they are split across POSIX threads only so that
 * the oracle can be timed on all host cores.  Each row is still a plain
 * qsort.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FLAG_SEQ_CLAMPED 1u  /* some seq_len > max_seq_len        */
#define ORACLE_FLAG_SEQ_NEGATIVE 2u /* some seq_len < 0 (treated as 0)   */

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -4

typedef struct {
    float v;
    int32_t i;
} entry_t;

static uint32_t float_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return u;
}

/* 2: NaN with sign clear, 1: any number (incl. +-inf, +-0), 0: NaN with sign set. */
static int value_class(float x) {
    if (!isnan(x)) return 1;
    return (float_bits(x) >> 31) ? 0 : 2;
}

/* > 0 if a ranks above b, < 0 if below, 0 if they tie. */
static int rank_compare(float a, float b) {
    int ca = value_class(a), cb = value_class(b);
    if (ca != cb) return ca > cb ? 1 : -1;
    if (ca == 1) {
#ifdef ORACLE_MUTATION_SIGNED_ZERO
        /* planted mistake: -0.0 ranks below +0.0 */
        if (a == 0.0f && b == 0.0f) {
            int sa = (int)(float_bits(a) >> 31), sb = (int)(float_bits(b) >> 31);
            if (sa != sb) return sa ? -1 : 1;
        }
#endif
        if (a > b) return 1;
        if (a < b) return -1;
        return 0;
    }
    uint32_t ua = float_bits(a), ub = float_bits(b);
    if (ua == ub) return 0;
    if (ca == 2) return ua > ub ? 1 : -1;
#ifdef ORACLE_MUTATION_NAN_PAYLOAD
    return ua > ub ? 1 : -1; /* planted mistake: negative NaNs ordered like positive ones */
#else
    return ua < ub ? 1 : -1;
#endif
}

/* qsort comparator: negative when x must come first (ranks higher). */
static int entry_order(const void* pa, const void* pb) {
    const entry_t* x = (const entry_t*)pa;
    const entry_t* y = (const entry_t*)pb;
    int r = rank_compare(x->v, y->v);
#ifdef ORACLE_MUTATION_ASCENDING
    r = -r; /* planted mistake: selects the smallest scores */
#endif
    if (r != 0) return r > 0 ? -1 : 1;
#ifdef ORACLE_MUTATION_TIE_LARGER_INDEX
    return x->i < y->i ? 1 : (x->i > y->i ? -1 : 0); /* planted mistake */
#else
    return x->i < y->i ? -1 : (x->i > y->i ? 1 : 0);
#endif
}

/* The page-table transform of one raw position (PR #26788, "Motivation"). */
static int32_t page_map(const int32_t* pt_row, int32_t page_size, int32_t raw) {
    if (raw < 0) return -1;
    uint32_t page = (uint32_t)pt_row[raw / page_size];
#ifdef ORACLE_MUTATION_PAGE_OFFSET
    uint32_t v = page * (uint32_t)page_size + (uint32_t)(raw % page_size) + 1u; /* planted mistake */
#else
    uint32_t v = page * (uint32_t)page_size + (uint32_t)(raw % page_size);
#endif
    return (int32_t)v;
}

static int32_t effective_len(int32_t s, int32_t max_seq_len, uint32_t* flags) {
    if (s < 0) {
        *flags |= ORACLE_FLAG_SEQ_NEGATIVE;
        return 0;
    }
    if (s > max_seq_len) {
        *flags |= ORACLE_FLAG_SEQ_CLAMPED;
        return max_seq_len;
    }
    return s;
}

typedef struct {
    const float* scores;
    int64_t row_stride;
    const int32_t* seq_lens;
    int32_t max_seq_len;
    const int32_t* page_table;
    int64_t pt_stride;
    int32_t page_size;
    int32_t k;
    int32_t* out;
    int32_t* raw_out;
    int32_t row_begin, row_end;
    uint32_t flags;
    int status;
} job_t;

static void* run_rows(void* arg) {
    job_t* job = (job_t*)arg;
    int64_t cap = 0;
    entry_t* buf = NULL;
    for (int32_t b = job->row_begin; b < job->row_end; ++b) {
        int32_t L = effective_len(job->seq_lens[b], job->max_seq_len, &job->flags);
        if (L > cap) {
            free(buf);
            buf = (entry_t*)malloc((size_t)L * sizeof(entry_t));
            if (!buf) {
                job->status = ORACLE_ENOMEM;
                return NULL;
            }
            cap = L;
        }
        const float* row = job->scores + (int64_t)b * job->row_stride;
        for (int32_t i = 0; i < L; ++i) {
            buf[i].v = row[i];
            buf[i].i = i;
        }
        if (L > 1) qsort(buf, (size_t)L, sizeof(entry_t), entry_order);
#ifdef ORACLE_MUTATION_NO_CLAMP_COUNT
        int32_t n = job->k; /* planted mistake: ignores short rows */
        if (n > L) n = L > 0 ? L : 0;
        if (L > 0 && L < job->k) n = L - 1;
#else
        int32_t n = job->k < L ? job->k : L;
#endif
        const int32_t* pt_row = job->page_table + (int64_t)b * job->pt_stride;
        int32_t* o = job->out + (int64_t)b * job->k;
        int32_t* r = job->raw_out ? job->raw_out + (int64_t)b * job->k : NULL;
        for (int32_t j = 0; j < job->k; ++j) {
            int32_t raw = j < n ? buf[j].i : -1;
            o[j] = page_map(pt_row, job->page_size, raw);
            if (r) r[j] = raw;
        }
    }
    free(buf);
    return NULL;
}

static int is_pow2(int32_t x) { return x > 0 && (x & (x - 1)) == 0; }

/*
 * Full top-k + transform over a batch.  All pointers are host memory.
 * out / raw_out: [batch, k] int32, row-major; raw_out may be NULL.
 * Output slot order within a row is the sort order (best first); callers that
 * compare with another implementation compare the sets.
 * Returns ORACLE_OK, ORACLE_EINVAL on bad arguments, ORACLE_ENOMEM.
 * *flags_out (may be NULL) receives ORACLE_FLAG_* bits.
 */
int oracle_topk_transform(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                          int32_t batch, int32_t max_seq_len, const int32_t* page_table,
                          int64_t page_table_stride, int32_t page_size, int32_t k, int32_t* out,
                          int32_t* raw_out, int32_t nthreads, uint32_t* flags_out) {
    if (batch < 0 || max_seq_len < 0 || k < 1 || !is_pow2(page_size) || row_stride < max_seq_len)
        return ORACLE_EINVAL;
    if (page_table_stride < ((int64_t)max_seq_len + page_size - 1) / page_size) return ORACLE_EINVAL;
    if (batch == 0) {
        if (flags_out) *flags_out = 0;
        return ORACLE_OK;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > batch) nthreads = batch;
    job_t* jobs = (job_t*)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return ORACLE_ENOMEM;
    }
    for (int32_t t = 0; t < nthreads; ++t) {
        job_t* j = &jobs[t];
        j->scores = scores;
        j->row_stride = row_stride;
        j->seq_lens = seq_lens;
        j->max_seq_len = max_seq_len;
        j->page_table = page_table;
        j->pt_stride = page_table_stride;
        j->page_size = page_size;
        j->k = k;
        j->out = out;
        j->raw_out = raw_out;
        j->row_begin = (int32_t)(((int64_t)batch * t) / nthreads);
        j->row_end = (int32_t)(((int64_t)batch * (t + 1)) / nthreads);
    }
    char* started = (char*)calloc((size_t)nthreads, 1);
    for (int32_t t = 1; t < nthreads; ++t) {
        if (started && pthread_create(&tids[t], NULL, run_rows, &jobs[t]) == 0) started[t] = 1;
        else run_rows(&jobs[t]); /* no thread available: run it here */
    }
    run_rows(&jobs[0]);
    uint32_t flags = jobs[0].flags;
    int status = jobs[0].status;
    for (int32_t t = 1; t < nthreads; ++t) {
        if (started && started[t]) pthread_join(tids[t], NULL);
        flags |= jobs[t].flags;
        if (jobs[t].status != ORACLE_OK) status = jobs[t].status;
    }
    free(started);
    free(jobs);
    free(tids);
    if (flags_out) *flags_out = flags;
    return status;
}

/*
 * The page-table transform alone, for raw positions that another step has
 * already selected: out[b][j] = page_map(raw[b][j]), -1 stays -1.
 */
int oracle_page_transform(const int32_t* raw, int32_t batch, int32_t k, const int32_t* page_table,
                          int64_t page_table_stride, int32_t page_size, int32_t* out) {
    if (batch < 0 || k < 1 || !is_pow2(page_size)) return ORACLE_EINVAL;
    for (int32_t b = 0; b < batch; ++b) {
        const int32_t* pt_row = page_table + (int64_t)b * page_table_stride;
        for (int32_t j = 0; j < k; ++j)
            out[(int64_t)b * k + j] = page_map(pt_row, page_size, raw[(int64_t)b * k + j]);
    }
    return ORACLE_OK;
}

/*
 * Row classification of the plan step (PR #26788, commit "Dynamic dispatch
 * via the plan's cluster_threshold": rows longer than the threshold go to the
 * multi-block path, the rest to one block each).  Writes the effective
 * (clamped) length of every row and whether it is long (len > threshold).
 */
int oracle_plan_classify(const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                         int32_t long_threshold, int32_t* eff_len, int32_t* is_long,
                         uint32_t* flags_out) {
    if (batch < 0 || max_seq_len < 0) return ORACLE_EINVAL;
    uint32_t flags = 0;
    for (int32_t b = 0; b < batch; ++b) {
        int32_t L = effective_len(seq_lens[b], max_seq_len, &flags);
        eff_len[b] = L;
        is_long[b] = L > long_threshold ? 1 : 0;
    }
    if (flags_out) *flags_out = flags;
    return ORACLE_OK;
}
