/*
 * pa_oracle.c -- plain, slow float64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load this library. The product (the CUDA library) never
 * calls it, includes it, or shares a line of code with it.
 *
 * What it computes, written straight from the definitions on the pages:
 *
 *   attention of one new token      Month 2 · PagedAttention (infra learning
 *                                    path), §2.1: attn = softmax(Q_i K_{:i}^T / sqrt(d)) V_{:i}
 *   K/V reached through a block table CS349E Lecture 7 notes, §4.1 (logical block
 *                                    i -> physical block); Month 2 · PagedAttention
 *                                    §5.2 (pool tensor of blocks) and §5.4 (the kernel
 *                                    looks up block_table[seq, logical_block])
 *   paging changes where K/V live,   CS349E Lecture 7 notes §4.2; CMU 15-779
 *   not the result                   Lecture 16 notes §3.3
 *
 * Readings fixed here (the pages leave them open):
 *   - pool layout is HND: cache[num_blocks][G][B][d]; token t of sequence s sits
 *     in physical block block_tables[s][t / B], row t % B;
 *   - query head h reads kv head h / (H / G) (contiguous GQA groups);
 *   - every t < context_lens[s] is attended (the new token included); the block
 *     count is ceil(ctx / B) -- the floor in the Month 2 §5.4 sketch would drop
 *     the partial last block;
 *   - the scale is an input (the pages use 1/sqrt(d));
 *   - an empty range gives m = -inf, l = 0, o = 0 (so ctx = 0 yields zeros).
 *
 * The softmax is the two-pass textbook form (max, then sum of exponentials),
 * not the online form the GPU uses. Stored 16-bit values are decoded from their
 * IEEE-754 / bfloat16 bit layouts below, in double precision, exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double pa_oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                    /* zero / subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);        /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE-754 binary32 (1 sign, 8 exponent with
 * bias 127, 7 fraction bits). */
double pa_oracle_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                   /* f * 2^-126 * 2^-7 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);        /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

static double load(const void *base, int64_t i, int dtype)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[i];
    if (dtype == ORACLE_F16)
        return pa_oracle_f16_to_f64(((const uint16_t *)base)[i]);
    return pa_oracle_bf16_to_f64(((const uint16_t *)base)[i]);
}

/* Attention of one query row over tokens [t0, t1) of one sequence.
 * Writes o[d] (normalised by l), *m (max score), *l (sum of exp(score - m)).
 * Returns 0, or 1 if a block id read from the table is outside the pool. */
static int attend_range(double *o, double *m_out, double *l_out,
                        const void *q, int64_t q_row, const void *k_cache, const void *v_cache,
                        int dtype, const int32_t *table, int t0, int t1,
                        int kv, int G, int d, int B, int64_t num_blocks, double scale)
{
    int n = t1 > t0 ? t1 - t0 : 0;
    for (int i = 0; i < d; i++)
        o[i] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (n == 0)
        return 0;

    double *z = (double *)malloc(sizeof(double) * (size_t)n);
    int64_t *row = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
    if (!z || !row) {
        free(z);
        free(row);
        return 2;
    }
    /* gather: the element offset of token t's row in the pool */
    for (int j = 0; j < n; j++) {
        int t = t0 + j;
        int64_t phys = table[t / B];
        if (phys < 0 || phys >= num_blocks) {
            free(z);
            free(row);
            return 1;
        }
        row[j] = ((phys * G + kv) * B + (t % B)) * (int64_t)d;
    }
    /* scores */
    for (int j = 0; j < n; j++) {
        double acc = 0.0;
        for (int i = 0; i < d; i++)
            acc += load(q, q_row * d + i, dtype) * load(k_cache, row[j] + i, dtype);
        z[j] = scale * acc;
    }
    /* softmax, pass 1: max */
    double m = -INFINITY;
    for (int j = 0; j < n; j++)
        if (z[j] > m)
            m = z[j];
    /* pass 2: weights and their sum */
    double l = 0.0;
    for (int j = 0; j < n; j++) {
        z[j] = exp(z[j] - m);
        l += z[j];
    }
    /* weighted sum of V rows */
    for (int j = 0; j < n; j++)
        for (int i = 0; i < d; i++)
            o[i] += z[j] * load(v_cache, row[j] + i, dtype);
    for (int i = 0; i < d; i++)
        o[i] /= l;
    *m_out = m;
    *l_out = l;
    free(z);
    free(row);
    return 0;
}

/*
 * out[S][H][d] (double) = attention of q[s][h] over the first context_lens[s]
 * tokens of sequence s. q, k_cache and v_cache hold `dtype` values (f32, or the
 * bit patterns of f16 / bf16). Returns 0 on success, 1 on a block id outside
 * [0, num_blocks), 3 on bad sizes.
 */
int pa_oracle_decode(double *out, const void *q, const void *k_cache, const void *v_cache,
                     int dtype, const int32_t *block_tables, int max_blocks,
                     const int32_t *context_lens, int S, int H, int G, int d, int B,
                     int64_t num_blocks, double scale, int num_threads)
{
    if (S < 0 || H <= 0 || G <= 0 || H % G || d <= 0 || B <= 0)
        return 3;
    int group = H / G;
    int bad = 0;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
#endif
    for (int64_t sh = 0; sh < (int64_t)S * H; sh++) {
        int s = (int)(sh / H), h = (int)(sh % H);
        int ctx = context_lens[s];
        if (ctx < 0 || (ctx + B - 1) / B > max_blocks) {
            bad |= 3;
            continue;
        }
        double m, l;
        bad |= attend_range(out + sh * d, &m, &l, q, sh, k_cache, v_cache, dtype,
                            block_tables + (int64_t)s * max_blocks, 0, ctx,
                            h / group, G, d, B, num_blocks, scale);
    }
    return bad;
}

/*
 * Per-partition softmax statistics: partition p of sequence s covers tokens
 * [p*T, min((p+1)*T, ctx)). For each (s, h, p):
 *   m[s][h][p] = max score, l[s][h][p] = sum exp(score - m),
 *   o[s][h][p][:] = sum exp(score - m) V / l.
 * P is the partition dimension of the output arrays (>= ceil(max ctx / T)).
 * Partitions past the end of a sequence get m = -inf, l = 0, o = 0.
 * This is the per-block form of attention the CS349E Lecture 7 notes §4.2 and
 * the CMU 15-779 Lecture 16 notes §3.3 describe, with blocks of T tokens.
 */
int pa_oracle_partitions(double *o, double *m, double *l, const void *q, const void *k_cache,
                         const void *v_cache, int dtype, const int32_t *block_tables,
                         int max_blocks, const int32_t *context_lens, int S, int H, int G, int d,
                         int B, int64_t num_blocks, double scale, int T, int P, int num_threads)
{
    if (S < 0 || H <= 0 || G <= 0 || H % G || d <= 0 || B <= 0 || T <= 0 || P <= 0)
        return 3;
    int group = H / G;
    int bad = 0;
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
#endif
    for (int64_t shp = 0; shp < (int64_t)S * H * P; shp++) {
        int64_t sh = shp / P;
        int p = (int)(shp % P);
        int s = (int)(sh / H), h = (int)(sh % H);
        int ctx = context_lens[s];
        if (ctx < 0 || (ctx + B - 1) / B > max_blocks || (ctx + T - 1) / T > P) {
            bad |= 3;
            continue;
        }
        int t0 = p * T, t1 = (p + 1) * T < ctx ? (p + 1) * T : ctx;
        bad |= attend_range(o + shp * d, m + shp, l + shp, q, sh, k_cache, v_cache, dtype,
                            block_tables + (int64_t)s * max_blocks, t0, t1,
                            h / group, G, d, B, num_blocks, scale);
    }
    return bad;
}

/*
 * Merge of per-partition results into the full attention, the rule the CMU
 * 15-779 Lecture 16 notes §3.3 call attention being "associative and
 * commutative": with M = max_p m_p and w_p = l_p exp(m_p - M),
 *   out = sum_p w_p o_p / sum_p w_p.
 * o is [R][P][d], m and l are [R][P]; out is [R][d]. Rows whose partitions are
 * all empty get zeros.
 */
void pa_oracle_merge(double *out, const double *o, const double *m, const double *l,
                     int64_t R, int P, int d)
{
    for (int64_t r = 0; r < R; r++) {
        double M = -INFINITY;
        for (int p = 0; p < P; p++)
            if (l[r * P + p] > 0.0 && m[r * P + p] > M)
                M = m[r * P + p];
        double wsum = 0.0;
        for (int i = 0; i < d; i++)
            out[r * d + i] = 0.0;
        for (int p = 0; p < P; p++) {
            double lp = l[r * P + p];
            if (!(lp > 0.0))
                continue;
            double w = lp * exp(m[r * P + p] - M);
            wsum += w;
            for (int i = 0; i < d; i++)
                out[r * d + i] += w * o[(r * P + p) * d + i];
        }
        if (wsum > 0.0)
            for (int i = 0; i < d; i++)
                out[r * d + i] /= wsum;
    }
}

int pa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
