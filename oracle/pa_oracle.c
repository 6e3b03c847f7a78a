/*
 * pa_oracle.c -- plain fp64 CPU oracle for paged-attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * reference that the CUDA path is checked against.  Only the test-suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product library never does, and this file shares no code, header,
 * table or helper with the CUDA sources.
 *
 * What it follows (sources are the web pages of the project_6 fork):
 *   - "paged_attention_v2_pytorch.py" commit list, commit 9cb7f9d
 *     ("PagedAttention V2 implementation"), section "Implementation":
 *       Phase 1, per (seq, head, partition): QK^T, softmax, weighted V sum;
 *                stores tmp_output, exp_sums, max_logits.
 *       Phase 2, cross-partition log-sum-exp reduction:
 *                global_max = max over partitions of max_logits,
 *                rescale    = exp(partition_max - global_max) * partition_exp_sum,
 *                output     = sum over partitions of (rescale / total_sum) * partition_output.
 *   - same page, commit 15ef28e ("Vectorize paged_attention_v2"), "Before":
 *       the per-block gather key_cache[physical_block] through the block table,
 *       and "Key changes": GQA by broadcasting one KV head over its query group.
 *   - "paged_attn.py" commit 490ff98, the summary_statistics paragraph:
 *       the {m, l, o} accumulator and its merge with factor exp(old_max - new_max).
 *
 * The decode result itself has a plain definition (the V2 phases reach it
 * exactly, up to rounding order): for sequence b and query head h with KV head
 * k = h / G (G = num_heads / num_kv_heads, contiguous groups),
 *     s_t   = scale * sum_d q[b,h,d] * K_t[d]             for t < seq_len[b]
 *     out   = sum_t softmax(s)_t * V_t
 * where K_t = key_cache[block_tables[b][t / bs], k, t % bs, :] (V likewise).
 * oracle_decode() writes exactly that out.  Subtracting max(s) inside the
 * exponent is an exact rewrite of softmax that only avoids overflow.
 *
 * Several new tokens per sequence (multi-query decode, q_len = Q >= 1): the
 * query is [S, Q, H, D] and query i of sequence b sits at position
 * L - Q + i, so it attends to the causal prefix t <= L - Q + i ("the
 * [kv_h, gqa, q_len, tile] batching" of the "paged_attn.py" commit 490ff98
 * online-softmax paragraph; the pages leave the mask implicit, and the
 * causal prefix is the reading taken).  A query that sees no token has a
 * zero output; a partition holding none of its visible tokens has
 * m_p = -inf, l_p = 0, o_p = 0 and contributes nothing to the merge.
 * Q = 1 is the single-query decode above.
 *
 * Storage types: query / key_cache / value_cache arrive as raw 16-bit
 * patterns (IEEE binary16 or bfloat16) and are decoded to double exactly by
 * this file's own bit decoding.  All arithmetic is in double.
 *
 * Threads: plain pthreads over the list of (seq, head) pairs.  No SIMD
 * intrinsics, so it builds and gives identical results on x86-64 and AArch64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2
#define ORACLE_EBLOCK 3 /* a block-table entry that is needed lies outside [0, num_blocks) */

/* ---------- exact decoding of 16-bit storage formats ---------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_binary16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^(1-15-10) */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac | 0x400), expo - 25); /* (1.frac) * 2^(e-15), 10 fraction bits */
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE binary32. */
static double decode_bfloat16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double decode16(uint16_t bits, int dtype)
{
    return dtype == ORACLE_BF16 ? decode_bfloat16(bits) : decode_binary16(bits);
}

double pa_oracle_decode_scalar(uint16_t bits, int dtype) { return decode16(bits, dtype); }

/* ---------- problem description ---------- */

typedef struct {
    const uint16_t *query;       /* [S, Q, H, D] */
    const uint16_t *key_cache;   /* [num_blocks, KV, bs, D] */
    const uint16_t *value_cache; /* [num_blocks, KV, bs, D] */
    const int32_t *block_tables; /* [S, max_blocks] */
    const int32_t *seq_lens;     /* [S] */
    int S, H, KV, D, num_blocks, bs, max_blocks;
    double scale;
    int dtype;
    int Q; /* new tokens per sequence */
} problem_t;

static int check_problem(const problem_t *p)
{
    if (!p->query || !p->key_cache || !p->value_cache || !p->block_tables || !p->seq_lens)
        return ORACLE_EINVAL;
    if (p->S <= 0 || p->H <= 0 || p->KV <= 0 || p->D <= 0 || p->bs <= 0 || p->num_blocks <= 0 ||
        p->max_blocks <= 0)
        return ORACLE_EINVAL;
    if (p->H % p->KV != 0 || p->Q < 1)
        return ORACLE_EINVAL;
    if (p->dtype != ORACLE_F16 && p->dtype != ORACLE_BF16)
        return ORACLE_EINVAL;
    for (int b = 0; b < p->S; ++b)
        if (p->seq_lens[b] < 0 || (int64_t)p->seq_lens[b] > (int64_t)p->max_blocks * p->bs)
            return ORACLE_EINVAL;
    return ORACLE_OK;
}

/* Pointer to row t of sequence b for KV head k, or NULL if the table entry is invalid. */
static const uint16_t *kv_row(const problem_t *p, const uint16_t *cache, int b, int k, int t)
{
    int32_t phys = p->block_tables[(int64_t)b * p->max_blocks + t / p->bs];
    if (phys < 0 || phys >= p->num_blocks)
        return NULL;
    return cache + (((int64_t)phys * p->KV + k) * p->bs + t % p->bs) * p->D;
}

/* Scaled logits s_t, t in [t0, t1), for query head h of sequence b. */
static int logits(const problem_t *p, int b, int h, int t0, int t1, const double *q, double *s)
{
    int k = h / (p->H / p->KV);
    for (int t = t0; t < t1; ++t) {
        const uint16_t *krow = kv_row(p, p->key_cache, b, k, t);
        if (!krow)
            return ORACLE_EBLOCK;
        double dot = 0.0;
        for (int d = 0; d < p->D; ++d)
            dot += q[d] * decode16(krow[d], p->dtype);
        s[t - t0] = p->scale * dot;
    }
    return ORACLE_OK;
}

/* Query row (sequence b, new token i) = r = b * Q + i. */
static void load_query(const problem_t *p, int r, int h, double *q)
{
    const uint16_t *qrow = p->query + ((int64_t)r * p->H + h) * p->D;
    for (int d = 0; d < p->D; ++d)
        q[d] = decode16(qrow[d], p->dtype);
}

/*
 * Softmax-weighted sum of V over tokens [t0, t1):
 *   m = max s,  w_t = exp(s_t - m),  l = sum w_t,  o = sum w_t V_t / l.
 * With [t0, t1) = [0, seq_len) this is the full decode output; with one
 * partition's range it is that partition's phase-1 result (o, l, m).
 */
static int softmax_v(const problem_t *p, int b, int h, int t0, int t1, const double *q, double *s,
                     double *o, double *m_out, double *l_out)
{
    int k = h / (p->H / p->KV);
    int rc = logits(p, b, h, t0, t1, q, s);
    if (rc)
        return rc;
    double m = -INFINITY;
    for (int t = 0; t < t1 - t0; ++t)
        if (s[t] > m)
            m = s[t];
    double l = 0.0;
    for (int d = 0; d < p->D; ++d)
        o[d] = 0.0;
    for (int t = t0; t < t1; ++t) {
        double w = exp(s[t - t0] - m);
        const uint16_t *vrow = kv_row(p, p->value_cache, b, k, t);
        if (!vrow)
            return ORACLE_EBLOCK;
        l += w;
        for (int d = 0; d < p->D; ++d)
            o[d] += w * decode16(vrow[d], p->dtype);
    }
    for (int d = 0; d < p->D; ++d)
        o[d] /= l;
    *m_out = m;
    *l_out = l;
    return ORACLE_OK;
}

/* ---------- thread pool over (seq, head) pairs ---------- */

typedef struct {
    const problem_t *p;
    const int32_t *pairs; /* [n, 2] (r, h), r = b * Q + i, or NULL for all S*Q*H in order */
    int n;
    int partition_size;   /* 0: full decode; >0: partition statistics */
    int max_partitions;   /* capacity of the per-pair partition arrays */
    double *out;          /* full decode: [n, D] */
    double *o_p;          /* partitions: [n, max_partitions, D] */
    double *m_p, *l_p;    /* partitions: [n, max_partitions] */
    int32_t *num_p;       /* partitions: [n] */
    int nthreads;
    int tid;
    int rc;
} job_t;

static void pair_at(const job_t *j, int i, int *r, int *h)
{
    if (j->pairs) {
        *r = j->pairs[2 * i];
        *h = j->pairs[2 * i + 1];
    } else {
        *r = i / j->p->H;
        *h = i % j->p->H;
    }
}

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    const problem_t *p = j->p;
    int64_t max_len = (int64_t)p->max_blocks * p->bs;
    double *q = (double *)malloc(sizeof(double) * p->D);
    double *s = (double *)malloc(sizeof(double) * (max_len > 0 ? max_len : 1));
    if (!q || !s) {
        j->rc = ORACLE_ENOMEM;
        goto done;
    }
    for (int i = j->tid; i < j->n; i += j->nthreads) {
        int r, h;
        pair_at(j, i, &r, &h);
        if (r < 0 || r >= p->S * p->Q || h < 0 || h >= p->H) {
            j->rc = ORACLE_EINVAL;
            goto done;
        }
        int b = r / p->Q;
        int L = p->seq_lens[b];
        /* tokens this query sees: t < visible, the causal prefix up to L - Q + i */
        int visible = L - p->Q + r % p->Q + 1;
        if (visible < 0)
            visible = 0;
        if (visible > L)
            visible = L;
        load_query(p, r, h, q);
        if (j->partition_size == 0) {
            double *dst = j->out + (int64_t)i * p->D;
            if (visible == 0) { /* no keys: defined as a zero output */
                for (int d = 0; d < p->D; ++d)
                    dst[d] = 0.0;
                continue;
            }
            double m, l;
            int rc = softmax_v(p, b, h, 0, visible, q, s, dst, &m, &l);
            if (rc) {
                j->rc = rc;
                goto done;
            }
        } else {
            int P = j->partition_size;
            int np = (int)((L + (int64_t)P - 1) / P);
            if (np > j->max_partitions) {
                j->rc = ORACLE_EINVAL;
                goto done;
            }
            j->num_p[i] = np;
            for (int part = 0; part < np; ++part) {
                int t0 = part * P;
                int t1 = t0 + P < L ? t0 + P : L;
                if (t1 > visible)
                    t1 = visible;
                int64_t slot = (int64_t)i * j->max_partitions + part;
                if (t1 <= t0) { /* none of this partition's tokens is visible */
                    j->m_p[slot] = -INFINITY;
                    j->l_p[slot] = 0.0;
                    for (int d = 0; d < p->D; ++d)
                        j->o_p[slot * p->D + d] = 0.0;
                    continue;
                }
                int rc = softmax_v(p, b, h, t0, t1, q, s, j->o_p + slot * p->D, &j->m_p[slot],
                                   &j->l_p[slot]);
                if (rc) {
                    j->rc = rc;
                    goto done;
                }
            }
        }
    }
done:
    free(q);
    free(s);
    return NULL;
}

static int run_jobs(job_t *proto, int nthreads)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > proto->n)
        nthreads = proto->n > 0 ? proto->n : 1;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return ORACLE_ENOMEM;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].nthreads = nthreads;
        jobs[t].tid = t;
        jobs[t].rc = ORACLE_OK;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0)
            break;
        started = t;
    }
    /* Any pair left without a thread is handled by re-running on this thread. */
    if (started < nthreads - 1) {
        for (int t = started + 1; t < nthreads; ++t)
            worker(&jobs[t]);
    }
    worker(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(th[t], NULL);
    int rc = ORACLE_OK;
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].rc)
            rc = jobs[t].rc;
    free(jobs);
    free(th);
    return rc;
}

/*
 * Full decode (the definition above).  pairs: [num_pairs, 2] of (b, h), or
 * NULL for every (b, h) in row-major order (num_pairs must then be S*H).
 * out: [num_pairs, D] doubles.  Returns 0 on success.
 */
int pa_oracle_decode_mq(const uint16_t *query, const uint16_t *key_cache,
                        const uint16_t *value_cache, const int32_t *block_tables,
                        const int32_t *seq_lens, int num_seqs, int q_len, int num_heads,
                        int num_kv_heads, int head_dim, int num_blocks, int block_size,
                        int max_blocks_per_seq, double scale, int dtype, const int32_t *pairs,
                        int num_pairs, double *out, int num_threads)
{
    problem_t p = {query, key_cache, value_cache, block_tables, seq_lens, num_seqs, num_heads,
                   num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq, scale, dtype,
                   q_len};
    int rc = check_problem(&p);
    if (rc)
        return rc;
    if (!out || num_pairs < 0 || (!pairs && num_pairs != num_seqs * q_len * num_heads))
        return ORACLE_EINVAL;
    job_t j;
    memset(&j, 0, sizeof j);
    j.p = &p;
    j.pairs = pairs;
    j.n = num_pairs;
    j.out = out;
    if (num_pairs == 0)
        return ORACLE_OK;
    return run_jobs(&j, num_threads);
}

int pa_oracle_decode(const uint16_t *query, const uint16_t *key_cache, const uint16_t *value_cache,
                     const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                     int num_heads, int num_kv_heads, int head_dim, int num_blocks, int block_size,
                     int max_blocks_per_seq, double scale, int dtype, const int32_t *pairs,
                     int num_pairs, double *out, int num_threads)
{
    return pa_oracle_decode_mq(query, key_cache, value_cache, block_tables, seq_lens, num_seqs, 1,
                               num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                               max_blocks_per_seq, scale, dtype, pairs, num_pairs, out,
                               num_threads);
}

/*
 * Phase 1 of the pages' V2, per (seq, head, partition): for partition
 * part = 0 .. ceil(L/P)-1 covering tokens [part*P, min(L, (part+1)*P)),
 *   m_p = max s_t,  l_p = sum exp(s_t - m_p),  o_p = sum exp(s_t - m_p) V_t / l_p.
 * Arrays are per pair with capacity max_partitions; num_p[i] receives the
 * partition count ceil(L/P) of pair i.  Entries past num_p[i] are untouched.
 */
int pa_oracle_partition_stats_mq(const uint16_t *query, const uint16_t *key_cache,
                                 const uint16_t *value_cache, const int32_t *block_tables,
                                 const int32_t *seq_lens, int num_seqs, int q_len, int num_heads,
                                 int num_kv_heads, int head_dim, int num_blocks, int block_size,
                                 int max_blocks_per_seq, double scale, int dtype,
                                 int partition_size, const int32_t *pairs, int num_pairs,
                                 int max_partitions, double *o_p, double *m_p, double *l_p,
                                 int32_t *num_p, int num_threads)
{
    problem_t p = {query, key_cache, value_cache, block_tables, seq_lens, num_seqs, num_heads,
                   num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq, scale, dtype,
                   q_len};
    int rc = check_problem(&p);
    if (rc)
        return rc;
    if (partition_size <= 0 || max_partitions <= 0 || !o_p || !m_p || !l_p || !num_p ||
        num_pairs < 0 || (!pairs && num_pairs != num_seqs * q_len * num_heads))
        return ORACLE_EINVAL;
    job_t j;
    memset(&j, 0, sizeof j);
    j.p = &p;
    j.pairs = pairs;
    j.n = num_pairs;
    j.partition_size = partition_size;
    j.max_partitions = max_partitions;
    j.o_p = o_p;
    j.m_p = m_p;
    j.l_p = l_p;
    j.num_p = num_p;
    if (num_pairs == 0)
        return ORACLE_OK;
    return run_jobs(&j, num_threads);
}

int pa_oracle_partition_stats(const uint16_t *query, const uint16_t *key_cache,
                              const uint16_t *value_cache, const int32_t *block_tables,
                              const int32_t *seq_lens, int num_seqs, int num_heads,
                              int num_kv_heads, int head_dim, int num_blocks, int block_size,
                              int max_blocks_per_seq, double scale, int dtype, int partition_size,
                              const int32_t *pairs, int num_pairs, int max_partitions, double *o_p,
                              double *m_p, double *l_p, int32_t *num_p, int num_threads)
{
    return pa_oracle_partition_stats_mq(query, key_cache, value_cache, block_tables, seq_lens,
                                        num_seqs, 1, num_heads, num_kv_heads, head_dim, num_blocks,
                                        block_size, max_blocks_per_seq, scale, dtype,
                                        partition_size, pairs, num_pairs, max_partitions, o_p, m_p,
                                        l_p, num_p, num_threads);
}

/*
 * Phase 2 of the pages' V2 for one (seq, head): the log-sum-exp merge of
 * num_partitions partial results o_p [num_partitions, D], m_p, l_p:
 *   global_max = max_p m_p
 *   rescale_p  = exp(m_p - global_max) * l_p
 *   total_sum  = sum_p rescale_p
 *   out        = sum_p (rescale_p / total_sum) * o_p
 * num_partitions == 0, or partitions that are all empty (l_p = 0), give a
 * zero output; an empty partition (m_p = -inf, l_p = 0) adds nothing.
 */
int pa_oracle_merge(const double *o_p, const double *m_p, const double *l_p, int num_partitions,
                    int head_dim, double *out)
{
    if (num_partitions < 0 || head_dim <= 0 || !out || (num_partitions > 0 && (!o_p || !m_p || !l_p)))
        return ORACLE_EINVAL;
    for (int d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (num_partitions == 0)
        return ORACLE_OK;
    double global_max = -INFINITY;
    for (int i = 0; i < num_partitions; ++i)
        if (m_p[i] > global_max)
            global_max = m_p[i];
    if (global_max == -INFINITY)
        return ORACLE_OK;
    double total_sum = 0.0;
    for (int i = 0; i < num_partitions; ++i)
        total_sum += exp(m_p[i] - global_max) * l_p[i];
    for (int i = 0; i < num_partitions; ++i) {
        if (l_p[i] == 0.0)
            continue;
        double weight = exp(m_p[i] - global_max) * l_p[i] / total_sum;
        for (int d = 0; d < head_dim; ++d)
            out[d] += weight * o_p[(int64_t)i * head_dim + d];
    }
    return ORACLE_OK;
}
