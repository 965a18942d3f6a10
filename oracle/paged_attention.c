/*
 * ORACLE -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow fp64 CPU statement of what paged decode attention computes.
 * Only the test suite, the package's smoke check and the benchmark's CPU
 * baseline load this file's library; the product path never does. It shares
 * no code, header, table or helper with the CUDA kernels.
 *
 * What it follows:
 *  - "What Does PagedAttention Actually Optimize?", section 17 (read_kv): a
 *    token position t lives in logical block t / B at offset t % B, and the
 *    block table maps that logical block to a physical block.
 *  - same page, section 8: Attention(Q, K, V) = softmax(Q K^T / sqrt(d)) V;
 *    paging changes where K and V live, not the result ("PagedAttention:
 *    KV cache virtual memory", section "Misconceptions").
 *  - grouped-query attention: query heads share KV heads ("PagedAttention,
 *    explained.", legend of the KV-size formula); query head h reads KV head
 *    h / (Hq / Hkv) (contiguous groups; the pages do not fix the mapping).
 *  - split into partitions and merged by log-sum-exp: the pages do not
 *    describe it; the plain definition is used -- each partition is ordinary
 *    softmax attention over its own tokens, reported as (max, sum of
 *    exponentials, normalised output), and the merge reweights partitions by
 *    sum * exp(max - global max).
 *
 * Method: rebuild each sequence's K and V contiguously (exact stored values
 * widened to double), then textbook softmax attention.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
static double widen(const void *base, int64_t idx, int kv_bf16)
{
    if (kv_bf16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

/* Gather KV head g of one sequence into dst[t][d], t < len, through its block
 * table. Returns -1 if a table entry the sequence needs is outside the pool. */
static int gather_head(double *dst, const void *cache, int kv_bf16, const int32_t *table,
                       int len, int block_size, int num_kv_heads, int head_dim, int g,
                       int num_blocks)
{
    for (int t = 0; t < len; ++t) {
        int logical = t / block_size;
        int offset = t % block_size;
        int64_t physical = table[logical];
        if (physical < 0 || physical >= num_blocks)
            return -1;
        int64_t row = ((physical * block_size + offset) * num_kv_heads + g) * (int64_t)head_dim;
        for (int d = 0; d < head_dim; ++d)
            dst[(int64_t)t * head_dim + d] = widen(cache, row + d, kv_bf16);
    }
    return 0;
}

/* Softmax attention of one query row over tokens [t0, t1) of a gathered head.
 * Writes the normalised output, the maximum scaled score and the sum of
 * exp(score - max). An empty range gives out = 0, max = -inf, sum = 0. */
static void attend(double *out, double *max_out, double *sum_out, const double *q,
                   const double *K, const double *V, int t0, int t1, int head_dim,
                   double scale, double *score)
{
    if (t1 <= t0) {
        for (int d = 0; d < head_dim; ++d)
            out[d] = 0.0;
        *max_out = -INFINITY;
        *sum_out = 0.0;
        return;
    }
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        double s = 0.0;
        for (int d = 0; d < head_dim; ++d)
            s += q[d] * K[(int64_t)t * head_dim + d];
        s *= scale;
        score[t - t0] = s;
        if (s > m)
            m = s;
    }
    double l = 0.0;
    for (int t = t0; t < t1; ++t)
        l += exp(score[t - t0] - m);
    for (int d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    for (int t = t0; t < t1; ++t) {
        double p = exp(score[t - t0] - m) / l;
        for (int d = 0; d < head_dim; ++d)
            out[d] += p * V[(int64_t)t * head_dim + d];
    }
    *max_out = m;
    *sum_out = l;
}

/*
 * Paged decode attention with the context of every sequence split into
 * partitions of `partition_size` tokens (partition_size <= 0: one partition
 * covering the whole context).
 *
 *   out       [B, Hq, P, D]  normalised output of each partition
 *   part_max  [B, Hq, P]     max scaled score of each partition (or NULL)
 *   part_sum  [B, Hq, P]     sum of exp(score - max) (or NULL)
 *   query     [B, Hq, D]     already widened to double
 *   k_cache, v_cache [num_blocks, block_size, Hkv, D] (fp32 or bf16 bits)
 *   block_tables [B, max_blocks], context_lens [B]
 *
 * Returns 0, or -1 on bad arguments / a table entry outside the pool.
 */
int oracle_paged_attention_partitions(double *out, double *part_max, double *part_sum,
                                      const double *query, const void *k_cache,
                                      const void *v_cache, int kv_bf16,
                                      const int32_t *block_tables, int max_blocks,
                                      const int32_t *context_lens, int num_seqs,
                                      int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int num_blocks, double scale,
                                      int partition_size, int num_partitions, int nthreads)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_heads % num_kv_heads != 0 || num_partitions <= 0)
        return -1;
    for (int b = 0; b < num_seqs; ++b) {
        if (context_lens[b] < 0 || context_lens[b] > max_blocks * block_size)
            return -1;
        if (partition_size > 0 && context_lens[b] > partition_size * num_partitions)
            return -1;
    }
    const int group = num_heads / num_kv_heads;
    int status = 0;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
    for (int unit = 0; unit < num_seqs * num_kv_heads; ++unit) {
        const int b = unit / num_kv_heads;
        const int g = unit % num_kv_heads;
        const int len = context_lens[b];
        const int64_t n = len > 0 ? len : 1;
        double *K = malloc(sizeof(double) * n * head_dim);
        double *V = malloc(sizeof(double) * n * head_dim);
        double *score = malloc(sizeof(double) * n);
        if (!K || !V || !score) {
#pragma omp atomic write
            status = -1;
            free(K); free(V); free(score);
            continue;
        }
        const int32_t *table = block_tables + (int64_t)b * max_blocks;
        if (gather_head(K, k_cache, kv_bf16, table, len, block_size, num_kv_heads, head_dim, g,
                        num_blocks) != 0 ||
            gather_head(V, v_cache, kv_bf16, table, len, block_size, num_kv_heads, head_dim, g,
                        num_blocks) != 0) {
#pragma omp atomic write
            status = -1;
            free(K); free(V); free(score);
            continue;
        }
        for (int h = g * group; h < (g + 1) * group; ++h) {
            const double *q = query + ((int64_t)b * num_heads + h) * head_dim;
            for (int p = 0; p < num_partitions; ++p) {
                int t0 = partition_size > 0 ? p * partition_size : 0;
                int t1 = partition_size > 0 ? (p + 1) * partition_size : len;
                if (t1 > len)
                    t1 = len;
                int64_t slot = ((int64_t)b * num_heads + h) * num_partitions + p;
                double m, l;
                attend(out + slot * head_dim, &m, &l, q, K, V, t0, t1, head_dim, scale, score);
                if (part_max)
                    part_max[slot] = m;
                if (part_sum)
                    part_sum[slot] = l;
            }
        }
        free(K);
        free(V);
        free(score);
    }
    return status;
}

/* Whole-context paged decode attention: out [B, Hq, D]. */
int oracle_paged_attention(double *out, const double *query, const void *k_cache,
                           const void *v_cache, int kv_bf16, const int32_t *block_tables,
                           int max_blocks, const int32_t *context_lens, int num_seqs,
                           int num_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, double scale, int nthreads)
{
    return oracle_paged_attention_partitions(out, NULL, NULL, query, k_cache, v_cache, kv_bf16,
                                             block_tables, max_blocks, context_lens, num_seqs,
                                             num_heads, num_kv_heads, head_dim, block_size,
                                             num_blocks, scale, 0, 1, nthreads);
}

/*
 * Log-sum-exp merge of partitions: with M = max_p part_max[p] and
 * w_p = part_sum[p] * exp(part_max[p] - M),
 *   out = sum_p w_p * part_out[p] / sum_p w_p.
 * Partitions with part_sum 0 (empty) carry no weight; a row whose partitions
 * are all empty is 0.
 */
int oracle_lse_merge(double *out, const double *part_out, const double *part_max,
                     const double *part_sum, int rows, int num_partitions, int head_dim)
{
    if (rows < 0 || num_partitions <= 0 || head_dim <= 0)
        return -1;
    for (int r = 0; r < rows; ++r) {
        const double *mx = part_max + (int64_t)r * num_partitions;
        const double *sm = part_sum + (int64_t)r * num_partitions;
        double M = -INFINITY;
        for (int p = 0; p < num_partitions; ++p)
            if (sm[p] > 0.0 && mx[p] > M)
                M = mx[p];
        double wsum = 0.0;
        double *o = out + (int64_t)r * head_dim;
        for (int d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        for (int p = 0; p < num_partitions; ++p) {
            if (!(sm[p] > 0.0))
                continue;
            double w = sm[p] * exp(mx[p] - M);
            wsum += w;
            const double *po = part_out + ((int64_t)r * num_partitions + p) * head_dim;
            for (int d = 0; d < head_dim; ++d)
                o[d] += w * po[d];
        }
        if (wsum > 0.0)
            for (int d = 0; d < head_dim; ++d)
                o[d] /= wsum;
    }
    return 0;
}
