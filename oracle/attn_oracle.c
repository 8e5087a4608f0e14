/*
 * attn_oracle.c -- plain fp64 CPU oracle for the causal grouped-query
 * attention forward pass computed as a streaming normalised sum.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes follows the header comment of the page
 * "Realization/Nvidia/SM86/StreamingAttentionSM86.alpha" (the forward pass of
 * softmax(Q K^T scale) V in base-2 units):
 *
 *   for query head h, compact K/V head g(h) = floor(h / (heads/kv_heads))
 *   (the page's grid mapping "head = kvHead * groups + z"), and row i:
 *     t_ij   = c * sum_e Q[h][i][e] * K[g][j][e]        for keys j <= i
 *     m_i    = max_j t_ij
 *     l_i    = sum_j 2^(t_ij - m_i)
 *     O[i][h*64 + e] = (sum_j 2^(t_ij - m_i) * VT[g][e][j]) / l_i
 *     LSE[h][i]      = m_i + log2 l_i                     (base 2)
 *
 * Layouts are the page's: Q [heads][T][64], K [kv_heads][T][64],
 * V^T [kv_heads][64][T] (binary16 bit patterns), O token-major
 * [T][heads*64], LSE [heads][T].  Everything here is fp64 from the exact
 * binary16 values; c is the binary32 value widened to fp64.  The method is
 * the plain two-pass definition (no streaming, no tiling), so it shares no
 * algorithm with the GPU kernel.  The diagonal key j = i is kept (the page's
 * diagonal-tile mask removes only columns beyond the row).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define HEAD_DIM 64

/* IEEE 754 binary16 bit pattern -> exact double. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* subnormal: mant * 2^-24 */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(mant | 0x400), expo - 25); /* (1024+mant) * 2^(e-25) */
    return sign ? -v : v;
}

static double g_half[65536];
static int g_half_ready = 0;

static void half_table_init(void)
{
    if (g_half_ready)
        return;
    for (int b = 0; b < 65536; ++b)
        g_half[b] = oracle_half_to_double((uint16_t)b);
    g_half_ready = 1;
}

static int check_shape(int64_t T, int64_t heads, int64_t kv_heads)
{
    if (T <= 0 || heads <= 0 || kv_heads <= 0)
        return -1;
    if (heads % kv_heads != 0)
        return -1;
    return 0;
}

/*
 * One output row: head h, query row i.  t is scratch of at least i+1
 * doubles.  o_row gets the 64 output values, *lse the base-2 log-sum-exp.
 */
static void oracle_row(const uint16_t *q, const uint16_t *k, const uint16_t *vT,
                       int64_t T, int64_t heads, int64_t kv_heads, double c,
                       int64_t h, int64_t i, double *t, double *o_row, double *lse)
{
    const int64_t group = heads / kv_heads;
    const int64_t g = h / group;
    const uint16_t *qi = q + (h * T + i) * HEAD_DIM;
    double qd[HEAD_DIM];
    for (int e = 0; e < HEAD_DIM; ++e)
        qd[e] = g_half[qi[e]];

    /* scores in base-2 units, keys 0..i */
    for (int64_t j = 0; j <= i; ++j) {
        const uint16_t *kj = k + (g * T + j) * HEAD_DIM;
        double s = 0.0;
        for (int e = 0; e < HEAD_DIM; ++e)
            s += qd[e] * g_half[kj[e]];
        t[j] = c * s;
    }

    /* row maximum, then the weights 2^(t - m) and their sum */
    double m = -INFINITY;
    for (int64_t j = 0; j <= i; ++j)
        if (t[j] > m)
            m = t[j];
    double l = 0.0;
    for (int64_t j = 0; j <= i; ++j) {
        t[j] = exp2(t[j] - m);
        l += t[j];
    }

    /* weighted sum of V's rows, normalised */
    for (int e = 0; e < HEAD_DIM; ++e) {
        const uint16_t *ve = vT + (g * HEAD_DIM + e) * T;
        double acc = 0.0;
        for (int64_t j = 0; j <= i; ++j)
            acc += t[j] * g_half[ve[j]];
        o_row[e] = acc / l;
    }
    *lse = m + log2(l);
}

static int resolve_threads(int threads)
{
#ifdef _OPENMP
    return threads > 0 ? threads : omp_get_max_threads();
#else
    (void)threads;
    return 1;
#endif
}

/* Number of threads the OpenMP runtime would use for threads <= 0. */
int oracle_max_threads(void)
{
    return resolve_threads(0);
}

/*
 * Selected rows: for n pairs (heads_idx[r], rows_idx[r]) write o[r][0..63]
 * and lse[r].  Returns 0, or -1 on a bad shape or index.
 */
int oracle_attn_fwd_rows(const uint16_t *q, const uint16_t *k, const uint16_t *vT,
                         int64_t T, int64_t heads, int64_t kv_heads, float c,
                         const int64_t *heads_idx, const int64_t *rows_idx, int64_t n,
                         double *o, double *lse, int threads)
{
    if (check_shape(T, heads, kv_heads))
        return -1;
    for (int64_t r = 0; r < n; ++r)
        if (heads_idx[r] < 0 || heads_idx[r] >= heads || rows_idx[r] < 0 || rows_idx[r] >= T)
            return -1;
    half_table_init();
    const double cd = (double)c;
    const int nt = resolve_threads(threads);
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nt)
#endif
    {
        double *t = (double *)malloc(sizeof(double) * (size_t)T);
        if (!t) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t r = 0; r < n; ++r)
            if (t)
                oracle_row(q, k, vT, T, heads, kv_heads, cd, heads_idx[r], rows_idx[r], t,
                           o + r * HEAD_DIM, lse + r);
        free(t);
    }
    (void)nt;
    return failed ? -1 : 0;
}

/*
 * Every row: o is [T][heads*64], lse is [heads][T].  Returns 0, or -1 on a
 * bad shape.
 */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *vT,
                    int64_t T, int64_t heads, int64_t kv_heads, float c,
                    double *o, double *lse, int threads)
{
    if (check_shape(T, heads, kv_heads))
        return -1;
    half_table_init();
    const double cd = (double)c;
    const int nt = resolve_threads(threads);
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nt)
#endif
    {
        double *t = (double *)malloc(sizeof(double) * (size_t)T);
        double row[HEAD_DIM];
        if (!t) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16) collapse(2)
#endif
        for (int64_t h = 0; h < heads; ++h)
            for (int64_t i = 0; i < T; ++i) {
                if (!t)
                    continue;
                double l2;
                oracle_row(q, k, vT, T, heads, kv_heads, cd, h, i, t, row, &l2);
                for (int e = 0; e < HEAD_DIM; ++e)
                    o[i * heads * HEAD_DIM + h * HEAD_DIM + e] = row[e];
                lse[h * T + i] = l2;
            }
        free(t);
    }
    (void)nt;
    return failed ? -1 : 0;
}
