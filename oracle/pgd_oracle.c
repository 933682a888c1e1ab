/*
 * Plain CPU oracle for single-token grouped-query attention over a paged
 * fp16 KV cache.  TEST INFRASTRUCTURE ONLY: the GPU library never links,
 * loads or calls this file; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg do.
 *
 * Everything here is written for a reader checking it against the pages
 * by eye: no blocking, no fusion, no reordering beyond what the definition
 * states, fp64 arithmetic throughout, OpenMP only across independent
 * (sequence, query head) pairs so the summation order of every output
 * element is fixed.
 *
 * Sources (page title, section):
 *   - "vllm-metal: hand-written Metal Paged Attention" (cf-1.com), section
 *     "What is Paged Attention": the KV cache is cut into fixed-size pages and
 *     a per-sequence page table (block_tables) maps logical page -> physical
 *     page.
 *   - same page, "Metal parallel model": work is split per
 *     (partition, KV head, sequence); the query heads that share one KV head
 *     form a group.
 *   - same page, "Four speed-up tricks", item 1: softmax in log2 space, log2(e)
 *     folded into the scale so every exponential is exp2; running max and
 *     exp-sum kept in one pass (online softmax).
 *   - same page, "Four speed-up tricks", item 4: long contexts are cut into
 *     256/512-token partitions; each partition writes a log2-space
 *     (max, exp-sum) pair plus its *normalised* partial output, and a
 *     separate reduce merges them.
 *   - "voxtral.c single-token attention" (dpshk.com), section "Single-token
 *     attention kernel": GQA with 32 query heads mapped onto 8 KV heads.
 *
 * Layouts (readings where the pages are silent):
 *   q            [S][Hq][D]           IEEE binary16 bit patterns
 *   k_cache      [NB][Hkv][BS][D]     IEEE binary16 bit patterns (the *_strided
 *   v_cache      [NB][Hkv][BS][D]      entry points take any row strides)
 *   block_tables [S][MB]              int32 physical page ids
 *   seq_lens     [S]                  int32, 0 <= L <= MB*BS
 *   out          [S][Hq][D]           fp64
 * Query head h reads KV head h / (Hq/Hkv) (integer division).
 * Token t of sequence s lives in physical page block_tables[s][t / BS],
 * row t % BS.  Page-table entries at or past ceil(L/BS) are never read.
 * A sequence of length 0 has an all-zero output row.
 *
 * Parity pins for every function are in tests/test_oracle.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Error codes returned by every entry point. */
#define ORC_OK 0
#define ORC_BAD_SHAPE 1      /* a size is non-positive or Hq % Hkv != 0 */
#define ORC_BAD_LENGTH 2     /* a sequence length is < 0 or > MB*BS      */
#define ORC_BAD_PAGE 3       /* a page id that must be read is outside [0, NB) */
#define ORC_NO_MEMORY 4

/* IEEE 754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0: subnormal, value = fraction * 2^-24;
 * exponent 31: infinity (fraction 0) or NaN;
 * otherwise value = (1024 + fraction) * 2^(exponent - 25). */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* Lookup table of all 65536 binary16 values, filled once from the
 * definition above (a cache of that function, nothing more). */
static double g_h2d[65536];
static int g_h2d_ready = 0;

static void h2d_init(void)
{
    if (g_h2d_ready)
        return;
    for (int i = 0; i < 65536; ++i)
        g_h2d[i] = oracle_half_to_double((uint16_t)i);
    g_h2d_ready = 1;
}

static int check_inputs(const int32_t *block_tables, const int32_t *seq_lens,
                        int S, int Hq, int Hkv, int D, int BS, int MB, int NB)
{
    if (S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || BS <= 0 || MB <= 0 || NB <= 0)
        return ORC_BAD_SHAPE;
    if (Hq % Hkv != 0)
        return ORC_BAD_SHAPE;
    for (int s = 0; s < S; ++s) {
        long L = seq_lens[s];
        if (L < 0 || L > (long)MB * BS)
            return ORC_BAD_LENGTH;
        long npages = (L + BS - 1) / BS;
        for (long j = 0; j < npages; ++j) {
            int32_t pp = block_tables[(long)s * MB + j];
            if (pp < 0 || pp >= NB)
                return ORC_BAD_PAGE;
        }
    }
    return ORC_OK;
}

/* Where the rows of a cache array are: the D values of token r of physical
 * page b, KV head g start at element b*page + g*head + r*token. */
typedef struct {
    long page, head, token;
} kv_strides;

/* The strides of the default layout [NB][Hkv][BS][D]. */
static kv_strides head_major(int Hkv, int BS, int D)
{
    kv_strides x = {(long)Hkv * BS * D, (long)BS * D, (long)D};
    return x;
}

/* Address of row t of sequence s, KV head g: page-table lookup
 * (cf-1.com, "What is Paged Attention"). */
static const uint16_t *kv_row(const uint16_t *cache, kv_strides x, const int32_t *block_tables,
                              int s, long t, int g, int BS, int MB)
{
    int32_t pp = block_tables[(long)s * MB + t / BS];
    return cache + pp * x.page + g * x.head + (t % BS) * x.token;
}

/* z_t = scale * sum_d qh[d] * k_t[d] for every token t < L of sequence s,
 * KV head g (qh: one query row of D values). */
static void logits(double *z, const uint16_t *qh, const uint16_t *k_cache, kv_strides x,
                   const int32_t *block_tables, double scale, int s, int g, long L, int D,
                   int BS, int MB)
{
    for (long t = 0; t < L; ++t) {
        const uint16_t *kt = kv_row(k_cache, x, block_tables, s, t, g, BS, MB);
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += g_h2d[qh[d]] * g_h2d[kt[d]];
        z[t] = scale * dot;
    }
}

/*
 * The definition: out[s][h] = sum_t w_t v_t with
 * w_t = exp(z_t - max z) / sum_u exp(z_u - max z).
 * (Natural exp; equal to the log2/exp2 form of the pages mathematically.)
 */
static int decode(double *out, const uint16_t *q, const uint16_t *k_cache,
                  const uint16_t *v_cache, kv_strides x, const int32_t *block_tables,
                  const int32_t *seq_lens, double scale, int S, int Hq, int Hkv, int D, int BS,
                  int MB, int NB, int num_threads)
{
    int rc = check_inputs(block_tables, seq_lens, S, Hq, Hkv, D, BS, MB, NB);
    if (rc)
        return rc;
    h2d_init();
    int G = Hq / Hkv;
    long pairs = (long)S * Hq;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads > 0 ? num_threads : 1)
    for (long sh = 0; sh < pairs; ++sh) {
        int s = (int)(sh / Hq), h = (int)(sh % Hq);
        int g = h / G;
        long L = seq_lens[s];
        double *o = out + sh * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        if (L == 0)
            continue;
        double *z = (double *)malloc(sizeof(double) * (size_t)L);
        if (!z) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        logits(z, q + sh * D, k_cache, x, block_tables, scale, s, g, L, D, BS, MB);
        double zmax = -INFINITY;
        for (long t = 0; t < L; ++t)
            if (z[t] > zmax)
                zmax = z[t];
        double den = 0.0;
        for (long t = 0; t < L; ++t)
            den += exp(z[t] - zmax);
        for (long t = 0; t < L; ++t) {
            double w = exp(z[t] - zmax) / den;
            const uint16_t *vt = kv_row(v_cache, x, block_tables, s, t, g, BS, MB);
            for (int d = 0; d < D; ++d)
                o[d] += w * g_h2d[vt[d]];
        }
        free(z);
    }
    return fail ? ORC_NO_MEMORY : ORC_OK;
}

int oracle_paged_gqa_decode(double *out, const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *block_tables,
                            const int32_t *seq_lens, double scale, int S, int Hq,
                            int Hkv, int D, int BS, int MB, int NB, int num_threads)
{
    return decode(out, q, k_cache, v_cache, head_major(Hkv, BS, D), block_tables, seq_lens,
                  scale, S, Hq, Hkv, D, BS, MB, NB, num_threads);
}

/* The definition over caches whose rows sit at the given strides (in
 * halves; every stride positive). */
int oracle_paged_gqa_decode_strided(double *out, const uint16_t *q, const uint16_t *k_cache,
                                    const uint16_t *v_cache, const int32_t *block_tables,
                                    const int32_t *seq_lens, double scale, int S, int Hq,
                                    int Hkv, int D, int BS, int MB, int NB, long page_stride,
                                    long head_stride, long token_stride, int num_threads)
{
    if (page_stride <= 0 || head_stride <= 0 || token_stride <= 0)
        return ORC_BAD_SHAPE;
    kv_strides x = {page_stride, head_stride, token_stride};
    return decode(out, q, k_cache, v_cache, x, block_tables, seq_lens, scale, S, Hq, Hkv, D,
                  BS, MB, NB, num_threads);
}

/*
 * Paged attention with several query tokens per sequence: the unified paged
 * variable-length attention of "vllm-metal" (introduction and "Three Metal
 * kernels": one kernel for prefill chunks, decode and the verification step
 * of speculative decoding).  Sequence s owns query rows cu_q[s] ..
 * cu_q[s+1]-1 of q ([total_q][Hq][D], total_q = cu_q[S]); its
 * n_s = cu_q[s+1] - cu_q[s] query tokens are the newest n_s of its
 * L_s = seq_lens[s] cached tokens (their K/V already in the cache), so query
 * i (0 <= i < n_s) sits at position L_s - n_s + i and attends every cached
 * token up to and including that position (causal).  For every query row r
 * and head h, with z_t = scale * q[r][h] . k_t over t = 0 .. pos:
 *   out[r][h] = sum_t w_t v_t,   w_t = exp(z_t - max z) / sum_u exp(z_u - max z).
 * A decode step is the case n_s = 1 for every sequence.  Caches are
 * addressed through strides as in oracle_paged_gqa_decode_strided.
 */
int oracle_paged_varlen(double *out, const uint16_t *q, const int32_t *cu_q,
                        const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, const int32_t *seq_lens, double scale,
                        int S, int Hq, int Hkv, int D, int BS, int MB, int NB, long page_stride,
                        long head_stride, long token_stride, int num_threads)
{
    int rc = check_inputs(block_tables, seq_lens, S, Hq, Hkv, D, BS, MB, NB);
    if (rc)
        return rc;
    if (page_stride <= 0 || head_stride <= 0 || token_stride <= 0 || cu_q[0] != 0)
        return ORC_BAD_SHAPE;
    for (int s = 0; s < S; ++s) {
        long n = (long)cu_q[s + 1] - cu_q[s];
        if (n < 0 || n > seq_lens[s])
            return ORC_BAD_LENGTH;
    }
    h2d_init();
    kv_strides x = {page_stride, head_stride, token_stride};
    int G = Hq / Hkv;
    long rows = (long)cu_q[S] * Hq;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads > 0 ? num_threads : 1)
    for (long rh = 0; rh < rows; ++rh) {
        long r = rh / Hq;
        int h = (int)(rh % Hq);
        int g = h / G;
        int s = 0;
        while (cu_q[s + 1] <= r) /* the sequence owning query row r */
            ++s;
        long n = (long)cu_q[s + 1] - cu_q[s];
        long pos = (long)seq_lens[s] - n + (r - cu_q[s]);
        long count = pos + 1; /* tokens 0 .. pos */
        double *o = out + rh * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        double *z = (double *)malloc(sizeof(double) * (size_t)count);
        if (!z) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        logits(z, q + rh * D, k_cache, x, block_tables, scale, s, g, count, D, BS, MB);
        double zmax = -INFINITY;
        for (long t = 0; t < count; ++t)
            if (z[t] > zmax)
                zmax = z[t];
        double den = 0.0;
        for (long t = 0; t < count; ++t)
            den += exp(z[t] - zmax);
        for (long t = 0; t < count; ++t) {
            double w = exp(z[t] - zmax) / den;
            const uint16_t *vt = kv_row(v_cache, x, block_tables, s, t, g, BS, MB);
            for (int d = 0; d < D; ++d)
                o[d] += w * g_h2d[vt[d]];
        }
        free(z);
    }
    return fail ? ORC_NO_MEMORY : ORC_OK;
}

/* Attention weights w_t of one (s, h), for the sum-to-one and closed-form
 * pins.  w must hold seq_lens[s] doubles. */
int oracle_attention_weights(double *w, const uint16_t *q, const uint16_t *k_cache,
                             const int32_t *block_tables, const int32_t *seq_lens,
                             double scale, int s, int h, int S, int Hq, int Hkv, int D,
                             int BS, int MB, int NB)
{
    int rc = check_inputs(block_tables, seq_lens, S, Hq, Hkv, D, BS, MB, NB);
    if (rc)
        return rc;
    if (s < 0 || s >= S || h < 0 || h >= Hq)
        return ORC_BAD_SHAPE;
    h2d_init();
    long L = seq_lens[s];
    if (L == 0)
        return ORC_OK;
    logits(w, q + ((long)s * Hq + h) * D, k_cache, head_major(Hkv, BS, D), block_tables, scale,
           s, h / (Hq / Hkv), L, D, BS, MB);
    double zmax = -INFINITY;
    for (long t = 0; t < L; ++t)
        if (w[t] > zmax)
            zmax = w[t];
    double den = 0.0;
    for (long t = 0; t < L; ++t)
        den += exp(w[t] - zmax);
    for (long t = 0; t < L; ++t)
        w[t] = exp(w[t] - zmax) / den;
    return ORC_OK;
}

/*
 * One-pass online softmax in log2 space, the order the pages describe
 * (cf-1.com, "Four speed-up tricks", item 1): scores are taken as
 * x_t = z_t * log2(e); a running max m and running exp2-sum l are carried
 * over the tokens; on a new max the sum and the accumulated output are
 * rescaled by exp2(m_old - m_new).
 */
int oracle_online_log2(double *out, const uint16_t *q, const uint16_t *k_cache,
                       const uint16_t *v_cache, const int32_t *block_tables,
                       const int32_t *seq_lens, double scale, int S, int Hq, int Hkv,
                       int D, int BS, int MB, int NB, int num_threads)
{
    int rc = check_inputs(block_tables, seq_lens, S, Hq, Hkv, D, BS, MB, NB);
    if (rc)
        return rc;
    h2d_init();
    int G = Hq / Hkv;
    const double log2e = 1.0 / log(2.0);
    kv_strides x = head_major(Hkv, BS, D);
    long pairs = (long)S * Hq;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads > 0 ? num_threads : 1)
    for (long sh = 0; sh < pairs; ++sh) {
        int s = (int)(sh / Hq), h = (int)(sh % Hq);
        int g = h / G;
        long L = seq_lens[s];
        double *o = out + sh * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        if (L == 0)
            continue;
        const uint16_t *qh = q + sh * D;
        double m = -INFINITY, l = 0.0;
        for (long t = 0; t < L; ++t) {
            const uint16_t *kt = kv_row(k_cache, x, block_tables, s, t, g, BS, MB);
            const uint16_t *vt = kv_row(v_cache, x, block_tables, s, t, g, BS, MB);
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += g_h2d[qh[d]] * g_h2d[kt[d]];
            double x = scale * dot * log2e;
            double m_new = x > m ? x : m;
            double alpha = exp2(m - m_new); /* exp2(-inf) = 0 on the first token */
            double p = exp2(x - m_new);
            l = alpha * l + p;
            for (int d = 0; d < D; ++d)
                o[d] = alpha * o[d] + p * g_h2d[vt[d]];
            m = m_new;
        }
        for (int d = 0; d < D; ++d)
            o[d] /= l;
    }
    return ORC_OK;
}

/*
 * Split-KV partials (cf-1.com, "Four speed-up tricks", item 4).
 * Partition p of sequence s covers logical tokens [p*P, min((p+1)*P, L)).
 * For every (s, h, p < ceil(L/P)), with x_t = z_t * log2(e):
 *   m[s][h][p]    = max_t x_t                       (log2-space max)
 *   l[s][h][p]    = sum_t exp2(x_t - m)             (exp-sum)
 *   o[s][h][p][:] = sum_t exp2(x_t - m) v_t / l     (normalised output)
 * Entries for p >= ceil(L/P) (up to NPmax) are m = -inf, l = 0, o = 0.
 * P may be any positive integer.
 */
int oracle_split_partials(double *m_out, double *l_out, double *o_out,
                          const uint16_t *q, const uint16_t *k_cache,
                          const uint16_t *v_cache, const int32_t *block_tables,
                          const int32_t *seq_lens, double scale, int S, int Hq, int Hkv,
                          int D, int BS, int MB, int NB, int P, int NPmax,
                          int num_threads)
{
    int rc = check_inputs(block_tables, seq_lens, S, Hq, Hkv, D, BS, MB, NB);
    if (rc)
        return rc;
    if (P <= 0 || NPmax <= 0)
        return ORC_BAD_SHAPE;
    for (int s = 0; s < S; ++s)
        if (((long)seq_lens[s] + P - 1) / P > NPmax)
            return ORC_BAD_SHAPE;
    h2d_init();
    int G = Hq / Hkv;
    const double log2e = 1.0 / log(2.0);
    kv_strides x = head_major(Hkv, BS, D);
    long pairs = (long)S * Hq;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads > 0 ? num_threads : 1)
    for (long sh = 0; sh < pairs; ++sh) {
        int s = (int)(sh / Hq), h = (int)(sh % Hq);
        int g = h / G;
        long L = seq_lens[s];
        for (int p = 0; p < NPmax; ++p) {
            m_out[sh * NPmax + p] = -INFINITY;
            l_out[sh * NPmax + p] = 0.0;
            for (int d = 0; d < D; ++d)
                o_out[(sh * NPmax + p) * D + d] = 0.0;
        }
        if (L == 0)
            continue;
        double *z = (double *)malloc(sizeof(double) * (size_t)L);
        if (!z) {
#pragma omp atomic write
            fail = 1;
            continue;
        }
        logits(z, q + sh * D, k_cache, x, block_tables, scale, s, g, L, D, BS, MB);
        long np = (L + P - 1) / P;
        for (long p = 0; p < np; ++p) {
            long t0 = p * P, t1 = t0 + P < L ? t0 + P : L;
            double m = -INFINITY;
            for (long t = t0; t < t1; ++t)
                if (z[t] * log2e > m)
                    m = z[t] * log2e;
            double l = 0.0;
            for (long t = t0; t < t1; ++t)
                l += exp2(z[t] * log2e - m);
            double *o = o_out + (sh * NPmax + p) * D;
            for (long t = t0; t < t1; ++t) {
                double w = exp2(z[t] * log2e - m);
                const uint16_t *vt = kv_row(v_cache, x, block_tables, s, t, g, BS, MB);
                for (int d = 0; d < D; ++d)
                    o[d] += w * g_h2d[vt[d]];
            }
            for (int d = 0; d < D; ++d)
                o[d] /= l;
            m_out[sh * NPmax + p] = m;
            l_out[sh * NPmax + p] = l;
        }
        free(z);
    }
    return fail ? ORC_NO_MEMORY : ORC_OK;
}

/*
 * Merge of the partition partials (the reduce of cf-1.com, "Four speed-up
 * tricks", item 4), per (s, h):
 *   M   = max_p m_p
 *   w_p = l_p * exp2(m_p - M)
 *   out = sum_p w_p o_p / sum_p w_p
 * Partitions with l_p = 0 (empty) are skipped; if all are empty the output
 * row is zero.
 */
int oracle_merge_partials(double *out, const double *m_in, const double *l_in,
                          const double *o_in, int S, int Hq, int D, int NPmax)
{
    if (S < 0 || Hq <= 0 || D <= 0 || NPmax <= 0)
        return ORC_BAD_SHAPE;
    long pairs = (long)S * Hq;
    for (long sh = 0; sh < pairs; ++sh) {
        double *o = out + sh * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        double M = -INFINITY;
        for (int p = 0; p < NPmax; ++p)
            if (l_in[sh * NPmax + p] > 0.0 && m_in[sh * NPmax + p] > M)
                M = m_in[sh * NPmax + p];
        if (M == -INFINITY)
            continue;
        double den = 0.0;
        for (int p = 0; p < NPmax; ++p) {
            double l = l_in[sh * NPmax + p];
            if (!(l > 0.0))
                continue;
            double w = l * exp2(m_in[sh * NPmax + p] - M);
            den += w;
            for (int d = 0; d < D; ++d)
                o[d] += w * o_in[(sh * NPmax + p) * D + d];
        }
        for (int d = 0; d < D; ++d)
            o[d] /= den;
    }
    return ORC_OK;
}

/*
 * The set of physical pages the method reads: for every (s, KV head g),
 * reads[s][g][j] = block_tables[s][j] for j < ceil(L/BS), and -1 for the
 * rest of the row (MB entries).  Every query head of the group reads the
 * same pages, so the set is per KV head.
 */
int oracle_page_reads(int32_t *reads, const int32_t *block_tables, const int32_t *seq_lens,
                      int S, int Hkv, int BS, int MB, int NB)
{
    int rc = check_inputs(block_tables, seq_lens, S, Hkv, Hkv, 1, BS, MB, NB);
    if (rc)
        return rc;
    for (int s = 0; s < S; ++s) {
        long npages = ((long)seq_lens[s] + BS - 1) / BS;
        for (int g = 0; g < Hkv; ++g)
            for (long j = 0; j < MB; ++j)
                reads[((long)s * Hkv + g) * MB + j] =
                    j < npages ? block_tables[(long)s * MB + j] : -1;
    }
    return ORC_OK;
}

/*
 * KV-cache append of a decode step: for every sequence s with L = seq_lens[s]
 * >= 1 and every KV head g, the newest token's key and value (k_new, v_new:
 * [S][Hkv][D]) are written at token L-1, i.e. row (L-1) % BS of physical page
 * block_tables[s][(L-1) / BS] (the page-table mapping of "vllm-metal", "What
 * is Paged Attention").  The caches are modified in place.  Sequences of
 * length 0 append nothing.
 */
static int append_kv(uint16_t *k_cache, uint16_t *v_cache, kv_strides x, const uint16_t *k_new,
                     const uint16_t *v_new, const int32_t *block_tables, const int32_t *seq_lens,
                     int S, int Hkv, int D, int BS, int MB, int NB)
{
    int rc = check_inputs(block_tables, seq_lens, S, Hkv, Hkv, D, BS, MB, NB);
    if (rc)
        return rc;
    for (int s = 0; s < S; ++s) {
        long L = seq_lens[s];
        if (L == 0)
            continue;
        int32_t pp = block_tables[(long)s * MB + (L - 1) / BS];
        for (int g = 0; g < Hkv; ++g) {
            long row = pp * x.page + g * x.head + ((L - 1) % BS) * x.token;
            for (int d = 0; d < D; ++d) {
                k_cache[row + d] = k_new[((long)s * Hkv + g) * D + d];
                v_cache[row + d] = v_new[((long)s * Hkv + g) * D + d];
            }
        }
    }
    return ORC_OK;
}

int oracle_append_kv(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k_new,
                     const uint16_t *v_new, const int32_t *block_tables, const int32_t *seq_lens,
                     int S, int Hkv, int D, int BS, int MB, int NB)
{
    return append_kv(k_cache, v_cache, head_major(Hkv, BS, D), k_new, v_new, block_tables,
                     seq_lens, S, Hkv, D, BS, MB, NB);
}

/* The append into caches whose rows sit at the given strides (in halves). */
int oracle_append_kv_strided(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k_new,
                             const uint16_t *v_new, const int32_t *block_tables,
                             const int32_t *seq_lens, int S, int Hkv, int D, int BS, int MB,
                             int NB, long page_stride, long head_stride, long token_stride)
{
    if (page_stride <= 0 || head_stride <= 0 || token_stride <= 0)
        return ORC_BAD_SHAPE;
    kv_strides x = {page_stride, head_stride, token_stride};
    return append_kv(k_cache, v_cache, x, k_new, v_new, block_tables, seq_lens, S, Hkv, D, BS,
                     MB, NB);
}

/*
 * Quantised KV pages in the affine group format of the Kapitsa series
 * (blog.hacking.pub, "权重怎样存储: 4-bit 编码与额外的量化参数"): a value is
 * approximated as scale * q + bias, with an unsigned integer code q and one
 * (scale, bias) pair per group of consecutive values, both stored as bf16.
 * Here the codes are 8-bit, a group is 64 consecutive head_dim elements of
 * one token row, and the pairs are stored [NB][Hkv][BS][D/64][2] next to the
 * codes [NB][Hkv][BS][D].
 */

/* bf16 -> double: the bf16 bits are the upper half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* w[i] = scale_g * codes[i] + bias_g for n values in groups of `group`
 * (meta: [n / group][2] bf16 pairs (scale, bias)). */
int oracle_dequant_affine(double *w, const uint8_t *codes, const uint16_t *meta, long n,
                          int group)
{
    if (n < 0 || group <= 0 || n % group != 0)
        return ORC_BAD_SHAPE;
    for (long i = 0; i < n; ++i) {
        long gidx = i / group;
        w[i] = oracle_bf16_to_double(meta[2 * gidx]) * codes[i] +
               oracle_bf16_to_double(meta[2 * gidx + 1]);
    }
    return ORC_OK;
}

/* The (scale, bias) pairs of the default layout [NB][Hkv][BS][D/64][2]. */
static kv_strides meta_head_major(int Hkv, int BS, int D)
{
    return head_major(Hkv, BS, (D / 64) * 2);
}

/* The decode definition over quantised caches: every K/V row is first
 * dequantised (oracle_dequant_affine), then attention as in
 * oracle_paged_gqa_decode (natural exp, fp64).  Row t of page b, KV head g:
 * codes at byte b*cx.page + g*cx.head + t*cx.token, its D/64 pairs at bf16
 * element b*mx.page + g*mx.head + t*mx.token. */
static int decode_q8(double *out, const uint16_t *q, const uint8_t *k_codes,
                     const uint16_t *k_meta, const uint8_t *v_codes, const uint16_t *v_meta,
                     kv_strides cx, kv_strides mx, const int32_t *block_tables,
                     const int32_t *seq_lens, double scale, int S, int Hq, int Hkv, int D, int BS,
                     int MB, int NB, int num_threads)
{
    int rc = check_inputs(block_tables, seq_lens, S, Hq, Hkv, D, BS, MB, NB);
    if (rc)
        return rc;
    if (D % 64 != 0)
        return ORC_BAD_SHAPE;
    h2d_init();
    int G = Hq / Hkv;
    long pairs = (long)S * Hq;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads > 0 ? num_threads : 1)
    for (long sh = 0; sh < pairs; ++sh) {
        int s = (int)(sh / Hq), h = (int)(sh % Hq);
        int g = h / G;
        long L = seq_lens[s];
        double *o = out + sh * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        if (L == 0)
            continue;
        double *z = (double *)malloc(sizeof(double) * (size_t)L);
        double *row = (double *)malloc(sizeof(double) * (size_t)D);
        if (!z || !row) {
            free(z);
            free(row);
#pragma omp atomic write
            fail = 1;
            continue;
        }
        const uint16_t *qh = q + sh * D;
        for (long t = 0; t < L; ++t) {
            long pp = block_tables[(long)s * MB + t / BS];
            oracle_dequant_affine(row, k_codes + pp * cx.page + g * cx.head + (t % BS) * cx.token,
                                  k_meta + pp * mx.page + g * mx.head + (t % BS) * mx.token, D,
                                  64);
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += g_h2d[qh[d]] * row[d];
            z[t] = scale * dot;
        }
        double zmax = -INFINITY;
        for (long t = 0; t < L; ++t)
            if (z[t] > zmax)
                zmax = z[t];
        double den = 0.0;
        for (long t = 0; t < L; ++t)
            den += exp(z[t] - zmax);
        for (long t = 0; t < L; ++t) {
            double w = exp(z[t] - zmax) / den;
            long pp = block_tables[(long)s * MB + t / BS];
            oracle_dequant_affine(row, v_codes + pp * cx.page + g * cx.head + (t % BS) * cx.token,
                                  v_meta + pp * mx.page + g * mx.head + (t % BS) * mx.token, D,
                                  64);
            for (int d = 0; d < D; ++d)
                o[d] += w * row[d];
        }
        free(z);
        free(row);
    }
    return fail ? ORC_NO_MEMORY : ORC_OK;
}

int oracle_paged_gqa_decode_q8(double *out, const uint16_t *q, const uint8_t *k_codes,
                               const uint16_t *k_meta, const uint8_t *v_codes,
                               const uint16_t *v_meta, const int32_t *block_tables,
                               const int32_t *seq_lens, double scale, int S, int Hq, int Hkv,
                               int D, int BS, int MB, int NB, int num_threads)
{
    return decode_q8(out, q, k_codes, k_meta, v_codes, v_meta, head_major(Hkv, BS, D),
                     meta_head_major(Hkv, BS, D), block_tables, seq_lens, scale, S, Hq, Hkv, D,
                     BS, MB, NB, num_threads);
}

/* The same over quantised caches in any layout: codes strides in bytes, the
 * pairs' strides in bf16 elements (every stride positive). */
int oracle_paged_gqa_decode_q8_strided(double *out, const uint16_t *q, const uint8_t *k_codes,
                                       const uint16_t *k_meta, const uint8_t *v_codes,
                                       const uint16_t *v_meta, const int32_t *block_tables,
                                       const int32_t *seq_lens, double scale, int S, int Hq,
                                       int Hkv, int D, int BS, int MB, int NB, long code_page,
                                       long code_head, long code_token, long meta_page,
                                       long meta_head, long meta_token, int num_threads)
{
    if (code_page <= 0 || code_head <= 0 || code_token <= 0 || meta_page <= 0 ||
        meta_head <= 0 || meta_token <= 0)
        return ORC_BAD_SHAPE;
    kv_strides cx = {code_page, code_head, code_token}, mx = {meta_page, meta_head, meta_token};
    return decode_q8(out, q, k_codes, k_meta, v_codes, v_meta, cx, mx, block_tables, seq_lens,
                     scale, S, Hq, Hkv, D, BS, MB, NB, num_threads);
}

/* ---------------------------------------------------------------- quantiser
 * Writing rows into quantised pages.  The pages give the affine format from
 * the reading side only (Kapitsa part 02, the affine group-64 weight format:
 * w ~ scale * q + bias, worked example scale 0.25, bias -1, q = [0, 3, 8, 15]
 * -> [-1, -0.25, 1, 2.75]); how scale and bias are chosen is not stated.  The
 * plainest reading for unsigned 8-bit codes: per group of 64 values the bias
 * is the group's minimum and the scale spreads the range over 255 steps,
 * both rounded to bf16 (nearest, ties to even) as they are stored, and each
 * code is the nearest step from the stored bias:
 *     mn = min x,  mx = max x                       (binary32)
 *     S  = bf16((mx - mn) / 255),  B = bf16(mn)
 *     q  = S > 0 ? clamp(rint((x - B) / S), 0, 255) : 0
 * Every step is one correctly rounded binary32 operation (this file is built
 * without contraction into fused multiply-adds), so any implementation that
 * takes the same steps in binary32 decides the same codes.
 */

/* binary32 -> bf16, round to nearest, ties to even (the upper 16 bits after
 * adding half an ulp of the result, plus one when the kept lsb is odd). */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays a (quiet) NaN */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* One group of n binary16 values -> n codes and the (scale, bias) pair. */
static void quantise_group(uint8_t *codes, uint16_t *pair, const uint16_t *x, int n)
{
    float mn = INFINITY, mx = -INFINITY;
    for (int i = 0; i < n; ++i) {
        float v = (float)g_h2d[x[i]]; /* exact: binary16 values are binary32 values */
        if (v < mn)
            mn = v;
        if (v > mx)
            mx = v;
    }
    float range = mx - mn;
    uint16_t sb = f32_to_bf16_rne(range / 255.0f), bb = f32_to_bf16_rne(mn);
    float S = bf16_to_f32(sb), B = bf16_to_f32(bb);
    for (int i = 0; i < n; ++i) {
        int q = 0;
        if (S > 0.0f) {
            float diff = (float)g_h2d[x[i]] - B;
            float t = rintf(diff / S);
            q = t < 0.0f ? 0 : (t > 255.0f ? 255 : (int)t);
        }
        codes[i] = (uint8_t)q;
    }
    pair[0] = sb;
    pair[1] = bb;
}

/* n binary16 values (n a multiple of `group`) -> codes [n] and pairs
 * [n / group][2] (scale, bias). */
int oracle_quantise_affine(uint8_t *codes, uint16_t *pairs, const uint16_t *x, long n, int group)
{
    if (n < 0 || group <= 0 || n % group != 0)
        return ORC_BAD_SHAPE;
    h2d_init();
    for (long gi = 0; gi < n / group; ++gi)
        quantise_group(codes + gi * group, pairs + 2 * gi, x + gi * group, group);
    return ORC_OK;
}

/* Rows src[n][h][:] (binary16, [N][Hkv][D]) written into the quantised
 * head-major cache at cache row slots[n] (page * BS + row; negative: row
 * skipped): codes [NB][Hkv][BS][D], pairs [NB][Hkv][BS][D/64][2]. */
static int quantise_rows(uint8_t *codes, uint16_t *meta, kv_strides cx, kv_strides mx,
                         const uint16_t *src, const int32_t *slots, int N, int Hkv, int D,
                         int BS, int NB)
{
    if (N < 0 || Hkv <= 0 || D <= 0 || D % 64 != 0 || BS <= 0 || NB <= 0)
        return ORC_BAD_SHAPE;
    h2d_init();
    for (int n = 0; n < N; ++n) {
        if (slots[n] < 0)
            continue;
        long page = slots[n] / BS, row = slots[n] % BS;
        if (page >= NB)
            return ORC_BAD_PAGE;
        for (int h = 0; h < Hkv; ++h) {
            uint8_t *c = codes + page * cx.page + h * cx.head + row * cx.token;
            uint16_t *m = meta + page * mx.page + h * mx.head + row * mx.token;
            for (int g = 0; g < D / 64; ++g)
                quantise_group(c + g * 64, m + 2 * g, src + ((long)n * Hkv + h) * D + g * 64, 64);
        }
    }
    return ORC_OK;
}

int oracle_quantise_rows(uint8_t *codes, uint16_t *meta, const uint16_t *src,
                         const int32_t *slots, int N, int Hkv, int D, int BS, int NB)
{
    return quantise_rows(codes, meta, head_major(Hkv, BS, D), meta_head_major(Hkv, BS, D), src,
                         slots, N, Hkv, D, BS, NB);
}

/* The decode step's append into quantised pages: sequence s's newest token
 * (position L_s - 1, L_s > 0) gets k_new[s] / v_new[s] ([S][Hkv][D]
 * binary16) written, quantised, into its row of page
 * block_tables[s][(L_s - 1) / BS]; the decode then reads them like every
 * other row (oracle_paged_gqa_decode_q8). */
static int append_kv_q8(uint8_t *k_codes, uint16_t *k_meta, uint8_t *v_codes, uint16_t *v_meta,
                        kv_strides cx, kv_strides mx, const uint16_t *k_new,
                        const uint16_t *v_new, const int32_t *block_tables,
                        const int32_t *seq_lens, int S, int Hkv, int D, int BS, int MB, int NB)
{
    if (S < 0 || MB <= 0)
        return ORC_BAD_SHAPE;
    int32_t *slots = (int32_t *)malloc(sizeof(int32_t) * (size_t)(S > 0 ? S : 1));
    if (!slots)
        return ORC_NO_MEMORY;
    int rc = ORC_OK;
    for (int s = 0; s < S && !rc; ++s) {
        long L = seq_lens[s];
        if (L < 0 || L > (long)MB * BS)
            rc = ORC_BAD_LENGTH;
        else if (L == 0)
            slots[s] = -1;
        else {
            int32_t page = block_tables[(long)s * MB + (L - 1) / BS];
            if (page < 0 || page >= NB)
                rc = ORC_BAD_PAGE;
            else
                slots[s] = (int32_t)(page * (long)BS + (L - 1) % BS);
        }
    }
    if (!rc)
        rc = quantise_rows(k_codes, k_meta, cx, mx, k_new, slots, S, Hkv, D, BS, NB);
    if (!rc)
        rc = quantise_rows(v_codes, v_meta, cx, mx, v_new, slots, S, Hkv, D, BS, NB);
    free(slots);
    return rc;
}

int oracle_append_kv_q8(uint8_t *k_codes, uint16_t *k_meta, uint8_t *v_codes, uint16_t *v_meta,
                        const uint16_t *k_new, const uint16_t *v_new, const int32_t *block_tables,
                        const int32_t *seq_lens, int S, int Hkv, int D, int BS, int MB, int NB)
{
    return append_kv_q8(k_codes, k_meta, v_codes, v_meta, head_major(Hkv, BS, D),
                        meta_head_major(Hkv, BS, D), k_new, v_new, block_tables, seq_lens, S,
                        Hkv, D, BS, MB, NB);
}

/* The append into quantised caches in any layout (strides as in
 * oracle_paged_gqa_decode_q8_strided). */
int oracle_append_kv_q8_strided(uint8_t *k_codes, uint16_t *k_meta, uint8_t *v_codes,
                                uint16_t *v_meta, const uint16_t *k_new, const uint16_t *v_new,
                                const int32_t *block_tables, const int32_t *seq_lens, int S,
                                int Hkv, int D, int BS, int MB, int NB, long code_page,
                                long code_head, long code_token, long meta_page, long meta_head,
                                long meta_token)
{
    if (code_page <= 0 || code_head <= 0 || code_token <= 0 || meta_page <= 0 ||
        meta_head <= 0 || meta_token <= 0)
        return ORC_BAD_SHAPE;
    kv_strides cx = {code_page, code_head, code_token}, mx = {meta_page, meta_head, meta_token};
    return append_kv_q8(k_codes, k_meta, v_codes, v_meta, cx, mx, k_new, v_new, block_tables,
                        seq_lens, S, Hkv, D, BS, MB, NB);
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
