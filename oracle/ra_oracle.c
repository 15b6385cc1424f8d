/*
 * Plain fp64 CPU oracle for blockwise exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled and called by the test
 * suite, by the smoke check and by the benchmark's CPU-baseline leg; no
 * product code path links it, loads it or falls back to it.  It shares no
 * code, header or constant with the CUDA library.
 *
 * What it computes is the plain definition of exact self-attention, which
 * ring attention reproduces without approximation:
 *   - "Ring Attention" glossary page (ultralytics.com/tr), section
 *     "Halka Dikkati Nasil Calisir": after N ring steps every query block has
 *     met every key/value block, and the four-device simulation is checked
 *     against the full expression softmax(q k^T / sqrt(dim)) v.
 *   - "Context Parallelism" glossary page (ultralytics.com/tr), section
 *     "Baglam Paralelligi Nasil Calisir?": the final result is mathematically
 *     equal to full-sequence attention.
 *   - Same page, section "Pratik Kullanim ve Odunlesimler": the PyTorch
 *     example lays q, k, v out as [batch, heads, sequence, dim] and calls
 *     scaled_dot_product_attention with is_causal=True.
 *
 * For one query row (b, h, t) with kv head g = h / (H / Hkv):
 *   s_u   = (sum_c q[b,h,t,c] k[b,g,u,c]) / sqrt(d)   for every allowed key u
 *   m     = max_u s_u
 *   l     = sum_u exp(s_u - m)
 *   out_c = sum_u exp(s_u - m) v[b,g,u,c] / l
 *   lse   = m + ln(l)
 * Allowed keys: all u (non-causal) or u <= t (causal), further restricted to
 * key_mask[u] != 0 when a key mask is given (attention over a subset of keys,
 * which is what one ring step computes).  A row with no allowed key has
 * out = 0 and lse = -inf.
 *
 * Readings where the pages are silent (listed with the rest in the design
 * notes): lse is the natural log of the softmax denominator including the
 * max; grouped-query attention maps query head h to kv head h / (H / Hkv);
 * the causal mask compares natural token positions, diagonal included.
 *
 * Two passes per row (max, then sums), fp64 throughout, libm exp/log, one
 * OpenMP thread per row.  Inputs are fp32, bf16 (raw uint16 bits) or fp64
 * and are widened exactly to fp64.
 *
 * `fault` plants a deliberate mistake for the tests that prove the oracle's
 * pins are discriminating; it is always 0 outside those tests.
 *   1 drop the 1/sqrt(d) scale        2 causal mask u < t instead of u <= t
 *   3 kv head h % Hkv (wrong GQA map)  4 lse = ln(l) without the max
 *   5 values taken from k, not v       6 scores use q[t] . k[t] (row index slip)
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2

static double widen(const void *base, int dtype, int64_t idx)
{
    if (dtype == ORACLE_F64)
        return ((const double *)base)[idx];
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    /* bf16: the 16 stored bits are the top half of an IEEE binary32 */
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Returns 0 on success, 1 on bad arguments, 2 on allocation failure. */
int oracle_attention_rows(const void *q, const void *k, const void *v, int dtype,
                          int64_t B, int64_t H, int64_t Hkv, int64_t S, int64_t d,
                          int causal, const uint8_t *key_mask,
                          const int64_t *rows, int64_t n_rows,
                          double *out, double *lse, int fault)
{
    if (!q || !k || !v || !rows || !out || !lse)
        return 1;
    if (B < 1 || H < 1 || Hkv < 1 || S < 1 || d < 1 || H % Hkv != 0)
        return 1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64)
        return 1;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * S)
            return 1;

    const int64_t group = H / Hkv;
    const double scale = (fault == 1) ? 1.0 : 1.0 / sqrt((double)d);
    int failed = 0;

#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)S * sizeof(double));
        double *qrow = (double *)malloc((size_t)d * sizeof(double));
        double *acc = (double *)malloc((size_t)d * sizeof(double));
        if (!s || !qrow || !acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (!s || !qrow || !acc)
                continue;
            const int64_t row = rows[r];
            const int64_t t = row % S;
            const int64_t bh = row / S;
            const int64_t h = bh % H;
            const int64_t b = bh / H;
            const int64_t g = (fault == 3) ? (h % Hkv) : (h / group);
            const int64_t qbase = ((b * H + h) * S + t) * d;
            const int64_t kvbase = (b * Hkv + g) * S * d;
            const void *vals = (fault == 5) ? k : v;

            for (int64_t c = 0; c < d; ++c)
                qrow[c] = widen(q, dtype, qbase + c);

            /* pass 1: scores of the allowed keys and their maximum */
            double m = -INFINITY;
            int64_t n_allowed = 0;
            for (int64_t u = 0; u < S; ++u) {
                int allowed = 1;
                if (causal)
                    allowed = (fault == 2) ? (u < t) : (u <= t);
                if (key_mask && !key_mask[u])
                    allowed = 0;
                if (!allowed) {
                    s[u] = -INFINITY;
                    continue;
                }
                const int64_t ku = (fault == 6) ? t : u;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dot += qrow[c] * widen(k, dtype, kvbase + ku * d + c);
                s[u] = dot * scale;
                if (s[u] > m)
                    m = s[u];
                ++n_allowed;
            }

            double *o = out + r * d;
            if (n_allowed == 0) {
                for (int64_t c = 0; c < d; ++c)
                    o[c] = 0.0;
                lse[r] = -INFINITY;
                continue;
            }

            /* pass 2: softmax denominator and weighted values */
            double l = 0.0;
            for (int64_t c = 0; c < d; ++c)
                acc[c] = 0.0;
            for (int64_t u = 0; u < S; ++u) {
                if (s[u] == -INFINITY)
                    continue;
                const double p = exp(s[u] - m);
                l += p;
                for (int64_t c = 0; c < d; ++c)
                    acc[c] += p * widen(vals, dtype, kvbase + u * d + c);
            }
            for (int64_t c = 0; c < d; ++c)
                o[c] = acc[c] / l;
            lse[r] = (fault == 4) ? log(l) : m + log(l);
        }
        free(s);
        free(qrow);
        free(acc);
    }
    return failed ? 2 : 0;
}

/* Number of OpenMP threads the oracle will use (reported by the benchmark). */
int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}

/* Thread count for the oracle's parallel loops from now on (0 restores all
 * cores); the benchmark reports a one-core rate beside the all-core one. */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}
