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
 *
 * The backward pass of the same page (dQ, dK, dV from dO, the forward's O
 * and L) is further below.
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

/*
 * Backward pass, following the backward comment of the page
 * "Realization/Nvidia/SM86/StreamingAttentionSM86.alpha": with the forward's
 * base-2 log-sum-exp L and output O given,
 *
 *   P_ij  = 2^(c S_ij - L_i)          for keys j <= i   (S = Q K^T)
 *   dP_ij = sum_e dO_ie V_je          (dP = dO V^T)
 *   D_i   = sum_e dO_ie O_ie          (the row term)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = s sum_j dS_ij K_j,   dK_j = s sum_i dS_ij Q_i,   dV_j = sum_i P_ij dO_i
 *
 * with s the natural score scale; dK and dV are summed over the query heads
 * of each K/V head's group (the page's grouped-gradient reduce).  O and L are
 * taken as given (fp64 arrays), so the oracle follows the same inputs the
 * kernels get.  Layouts: dO and O token-major [T][heads*64]; L and D
 * [heads][T]; dQ [heads][T][64]; dK [kv_heads][T][64]; dV^T [kv_heads][64][T].
 */
static double dot64_hq(const uint16_t *a, const double *b)
{
    double s = 0.0;
    for (int e = 0; e < HEAD_DIM; ++e)
        s += g_half[a[e]] * b[e];
    return s;
}

/* D for every (head, row): D[h][i] = sum_e dO[i][h*64+e] O[i][h*64+e]. */
static void oracle_row_terms(const double *o, const uint16_t *dO, int64_t T, int64_t heads,
                             double *D)
{
    for (int64_t h = 0; h < heads; ++h)
        for (int64_t i = 0; i < T; ++i) {
            const uint16_t *g = dO + (i * heads + h) * HEAD_DIM;
            const double *oo = o + (i * heads + h) * HEAD_DIM;
            double s = 0.0;
            for (int e = 0; e < HEAD_DIM; ++e)
                s += g_half[g[e]] * oo[e];
            D[h * T + i] = s;
        }
}

/* dQ row i of head h (D for all rows given). */
static void oracle_dq_row(const uint16_t *q, const uint16_t *k, const uint16_t *vT,
                          const double *lse, const uint16_t *dO, const double *D,
                          int64_t T, int64_t heads, int64_t kv_heads, double c, double s,
                          int64_t h, int64_t i, double *out)
{
    const int64_t g = h / (heads / kv_heads);
    double qd[HEAD_DIM], gd[HEAD_DIM], acc[HEAD_DIM];
    for (int e = 0; e < HEAD_DIM; ++e) {
        qd[e] = g_half[q[(h * T + i) * HEAD_DIM + e]];
        gd[e] = g_half[dO[(i * heads + h) * HEAD_DIM + e]];
        acc[e] = 0.0;
    }
    for (int64_t j = 0; j <= i; ++j) {
        const uint16_t *kj = k + (g * T + j) * HEAD_DIM;
        const double p = exp2(c * dot64_hq(kj, qd) - lse[h * T + i]);
        double dp = 0.0;
        for (int e = 0; e < HEAD_DIM; ++e)
            dp += gd[e] * g_half[vT[(g * HEAD_DIM + e) * T + j]];
        const double ds = p * (dp - D[h * T + i]);
        for (int e = 0; e < HEAD_DIM; ++e)
            acc[e] += ds * g_half[kj[e]];
    }
    for (int e = 0; e < HEAD_DIM; ++e)
        out[e] = s * acc[e];
}

/* dK and dV rows j of K/V head g, summed over the group's query heads. */
static void oracle_dkv_row(const uint16_t *q, const uint16_t *k, const uint16_t *vT,
                           const double *lse, const uint16_t *dO, const double *D,
                           int64_t T, int64_t heads, int64_t kv_heads, double c, double s,
                           int64_t g, int64_t j, double *dk_out, double *dv_out)
{
    const int64_t group = heads / kv_heads;
    double kd[HEAD_DIM], vd[HEAD_DIM], dk[HEAD_DIM], dv[HEAD_DIM];
    for (int e = 0; e < HEAD_DIM; ++e) {
        kd[e] = g_half[k[(g * T + j) * HEAD_DIM + e]];
        vd[e] = g_half[vT[(g * HEAD_DIM + e) * T + j]];
        dk[e] = dv[e] = 0.0;
    }
    for (int64_t h = g * group; h < (g + 1) * group; ++h)
        for (int64_t i = j; i < T; ++i) {
            const uint16_t *qi = q + (h * T + i) * HEAD_DIM;
            const uint16_t *gi = dO + (i * heads + h) * HEAD_DIM;
            const double p = exp2(c * dot64_hq(qi, kd) - lse[h * T + i]);
            const double dp = dot64_hq(gi, vd);
            const double ds = p * (dp - D[h * T + i]);
            for (int e = 0; e < HEAD_DIM; ++e) {
                dk[e] += ds * g_half[qi[e]];
                dv[e] += p * g_half[gi[e]];
            }
        }
    for (int e = 0; e < HEAD_DIM; ++e) {
        dk_out[e] = s * dk[e];
        dv_out[e] = dv[e];
    }
}

/*
 * Full backward.  o: fp64 [T][heads*64]; lse: fp64 [heads][T]; dO: binary16
 * [T][heads*64].  Writes dq [heads][T][64], dk [kv_heads][T][64],
 * dvT [kv_heads][64][T] and D [heads][T].  Returns 0, or -1 on a bad shape.
 */
int oracle_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *vT, const double *o,
                    const double *lse, const uint16_t *dO, int64_t T, int64_t heads,
                    int64_t kv_heads, float c, float s, double *dq, double *dk, double *dvT,
                    double *D, int threads)
{
    if (check_shape(T, heads, kv_heads))
        return -1;
    half_table_init();
    oracle_row_terms(o, dO, T, heads, D);
    const double cd = (double)c, sd = (double)s;
    const int nt = resolve_threads(threads);
    (void)nt;
#ifdef _OPENMP
#pragma omp parallel num_threads(nt)
#endif
    {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16) collapse(2) nowait
#endif
        for (int64_t h = 0; h < heads; ++h)
            for (int64_t i = 0; i < T; ++i)
                oracle_dq_row(q, k, vT, lse, dO, D, T, heads, kv_heads, cd, sd, h, i,
                              dq + (h * T + i) * HEAD_DIM);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16) collapse(2)
#endif
        for (int64_t g = 0; g < kv_heads; ++g)
            for (int64_t j = 0; j < T; ++j) {
                double dkr[HEAD_DIM], dvr[HEAD_DIM];
                oracle_dkv_row(q, k, vT, lse, dO, D, T, heads, kv_heads, cd, sd, g, j, dkr, dvr);
                for (int e = 0; e < HEAD_DIM; ++e) {
                    dk[(g * T + j) * HEAD_DIM + e] = dkr[e];
                    dvT[(g * HEAD_DIM + e) * T + j] = dvr[e];
                }
            }
    }
    return 0;
}

/*
 * Sampled rows of the backward: n_q (head, row) pairs of dQ and n_kv
 * (kv_head, row) pairs of dK and dV.  Needs the row terms of every row, so
 * it computes D first (cheap: one dot product per row).  dq_out [n_q][64],
 * dk_out and dv_out [n_kv][64].  Returns 0, or -1 on a bad shape or index.
 */
int oracle_attn_bwd_rows(const uint16_t *q, const uint16_t *k, const uint16_t *vT,
                         const double *o, const double *lse, const uint16_t *dO, int64_t T,
                         int64_t heads, int64_t kv_heads, float c, float s,
                         const int64_t *qh, const int64_t *qi, int64_t n_q,
                         const int64_t *kg, const int64_t *kj, int64_t n_kv,
                         double *dq_out, double *dk_out, double *dv_out, int threads)
{
    if (check_shape(T, heads, kv_heads))
        return -1;
    for (int64_t r = 0; r < n_q; ++r)
        if (qh[r] < 0 || qh[r] >= heads || qi[r] < 0 || qi[r] >= T)
            return -1;
    for (int64_t r = 0; r < n_kv; ++r)
        if (kg[r] < 0 || kg[r] >= kv_heads || kj[r] < 0 || kj[r] >= T)
            return -1;
    half_table_init();
    double *D = (double *)malloc(sizeof(double) * (size_t)(heads * T));
    if (!D)
        return -1;
    oracle_row_terms(o, dO, T, heads, D);
    const double cd = (double)c, sd = (double)s;
    const int nt = resolve_threads(threads);
    (void)nt;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
    for (int64_t r = 0; r < n_q + n_kv; ++r) {
        if (r < n_q)
            oracle_dq_row(q, k, vT, lse, dO, D, T, heads, kv_heads, cd, sd, qh[r], qi[r],
                          dq_out + r * HEAD_DIM);
        else
            oracle_dkv_row(q, k, vT, lse, dO, D, T, heads, kv_heads, cd, sd, kg[r - n_q],
                           kj[r - n_q], dk_out + (r - n_q) * HEAD_DIM,
                           dv_out + (r - n_q) * HEAD_DIM);
    }
    free(D);
    return 0;
}

/*
 * ---------------------------------------------------------------------------
 * The fused QKV producer (the launches that make Q, K and V^T for the forward
 * pass): on the page ".../Coppelius/Build/Graph.alpha" a layer's attention
 * inputs come from the QKV product of the normed activations with the QKV
 * matrix (three parts), then "qk-rope" (rotary embedding of the query and key
 * heads with the cosine and sine tables: a row per position, a column per
 * head-dimension pair) and "value-transpose".  Written out, for token t:
 *
 *   y[t][n] = sum_i X[t][i] W[n][i]                  n < (heads + 2 kv_heads) * 64
 *
 * with the parts in the order Q (heads * 64 outputs), K (kv_heads * 64), V
 * (kv_heads * 64) and head h of a part at its outputs h*64 .. h*64 + 63.  Query
 * and key heads are rotated pair by pair: pair p of a head is its elements
 * (2p, 2p + 1), and with c = C[t][p], s = S[t][p]
 *
 *   (a, b) -> (a c - b s,  a s + b c).
 *
 * Outputs (fp64, unrounded): q [heads][T][64], k [kv_heads][T][64],
 * vT [kv_heads][64][T].  X and W are binary16 bit patterns, the tables
 * binary32; all arithmetic is fp64.
 */
int oracle_qkv_rope(const uint16_t *x, const uint16_t *w, const float *cos_tab,
                    const float *sin_tab, int64_t T, int64_t width, int64_t heads,
                    int64_t kv_heads, double *q, double *k, double *vT, int threads)
{
    if (T <= 0 || width <= 0 || heads <= 0 || kv_heads <= 0 || heads % kv_heads != 0)
        return -1;
    half_table_init();
    const int64_t n_out = (heads + 2 * kv_heads) * HEAD_DIM;
    const int nt = resolve_threads(threads);
    (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t t = 0; t < T; ++t) {
        double *y = (double *)malloc((size_t)n_out * sizeof(double));
        const uint16_t *xr = x + t * width;
        for (int64_t n = 0; n < n_out; ++n) {
            const uint16_t *wr = w + n * width;
            double acc = 0.0;
            for (int64_t i = 0; i < width; ++i)
                acc += g_half[xr[i]] * g_half[wr[i]];
            y[n] = acc;
        }
        for (int64_t hh = 0; hh < heads + kv_heads; ++hh) {      /* query heads, then key heads */
            const double *src = y + hh * HEAD_DIM;
            double *dst = hh < heads ? q + (hh * T + t) * HEAD_DIM
                                     : k + ((hh - heads) * T + t) * HEAD_DIM;
            for (int p = 0; p < HEAD_DIM / 2; ++p) {
                const double c = (double)cos_tab[t * (HEAD_DIM / 2) + p];
                const double s = (double)sin_tab[t * (HEAD_DIM / 2) + p];
                const double a = src[2 * p], b = src[2 * p + 1];
                dst[2 * p] = a * c - b * s;
                dst[2 * p + 1] = a * s + b * c;
            }
        }
        for (int64_t g = 0; g < kv_heads; ++g) {                  /* value heads, transposed */
            const double *src = y + (heads + kv_heads + g) * HEAD_DIM;
            for (int e = 0; e < HEAD_DIM; ++e)
                vT[(g * HEAD_DIM + e) * T + t] = src[e];
        }
        free(y);
    }
    return 0;
}
