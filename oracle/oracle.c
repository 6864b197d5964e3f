/*
 * oracle.c -- plain, slow, fp64 CPU statement of query-aware page selection
 * followed by masked attention over the selected pages.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path links,
 * loads or calls this file; only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or helper
 * with the CUDA path.
 *
 * Source of the method: "TinyServe: Query-Aware Cache Selection for Efficient
 * LLM Serving" (arXiv 2509.12211), section 方法详解 / 关键设计: every KV-cache
 * block carries a bounding box of what it contains; at decode time the query
 * is compared with every block's box and the blocks with the highest
 * similarity are loaded; the abstract adds that scoring, sparse memory access
 * and masked attention form one decode step.  The pages give no formula; the
 * readings used here are:
 *   - the box of page p is the per-channel minimum lo[p][c] and maximum
 *     hi[p][c] of the keys stored in its valid slots;
 *   - the similarity is the largest value q.k can take inside the box,
 *     sum_c max(q_c*lo_c, q_c*hi_c), maximised over the query heads that share
 *     the KV head (grouped-query attention);
 *   - the sink page (logical page 0) and the newest page (N-1) are always
 *     kept; the remaining budget goes to the highest scores, ties to the lower
 *     page index; a budget of at least N keeps every page;
 *   - attention is softmax(scale * q.k) over the tokens of the kept pages whose
 *     position is below the sequence length, times V, with scale = 1/sqrt(d).
 *
 * Every function works on ONE (sequence, KV head) with logical (not physical)
 * token order: K and V are [L][d] row-major, q is [G][d].  All arithmetic is
 * fp64.  No blocking, no fusion, no reordering beyond the definitions.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

static int num_pages_of(int L, int P) { return (L + P - 1) / P; }

/* Bounding box of every page, computed from scratch over its valid tokens.
 * lo, hi: [N][d] with N = ceil(L/P). */
void oracle_page_bounds(int L, int d, int P, const double *K, double *lo, double *hi)
{
    int N = num_pages_of(L, P);
    for (int p = 0; p < N; ++p) {
        int t0 = p * P, t1 = (p + 1) * P < L ? (p + 1) * P : L;
        for (int c = 0; c < d; ++c) {
            double mn = K[(size_t)t0 * d + c], mx = mn;
            for (int t = t0 + 1; t < t1; ++t) {
                double x = K[(size_t)t * d + c];
                if (x < mn) mn = x;
                if (x > mx) mx = x;
            }
            lo[(size_t)p * d + c] = mn;
            hi[(size_t)p * d + c] = mx;
        }
    }
}

/* The same boxes, maintained the way an append-time builder keeps them:
 * tokens arrive in chunks (chunk_lens sums to L); each chunk writes its tokens
 * into their slots and folds them into the box of their page; a page whose
 * slot 0 is written by the chunk starts a fresh box.  Independent of
 * oracle_page_bounds so the two can pin each other. */
void oracle_page_bounds_by_appends(int L, int d, int P, const double *K, int n_chunks,
                                   const int *chunk_lens, double *lo, double *hi)
{
    int pos = 0;
    for (int ch = 0; ch < n_chunks; ++ch) {
        for (int i = 0; i < chunk_lens[ch]; ++i, ++pos) {
            if (pos >= L) return;
            int p = pos / P, slot = pos % P;
            const double *k = K + (size_t)pos * d;
            double *l = lo + (size_t)p * d, *h = hi + (size_t)p * d;
            for (int c = 0; c < d; ++c) {
                if (slot == 0) {
                    l[c] = k[c];
                    h[c] = k[c];
                } else {
                    l[c] = fmin(l[c], k[c]);
                    h[c] = fmax(h[c], k[c]);
                }
            }
        }
    }
}

/* Score of every page: max over the G query heads of the largest q.k inside
 * the page's box.  s: [N]. */
void oracle_page_scores(int G, int d, int N, const double *q, const double *lo,
                        const double *hi, double *s)
{
    for (int p = 0; p < N; ++p) {
        double best = -INFINITY;
        for (int g = 0; g < G; ++g) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) {
                double a = q[(size_t)g * d + c] * lo[(size_t)p * d + c];
                double b = q[(size_t)g * d + c] * hi[(size_t)p * d + c];
                acc += a > b ? a : b;
            }
            if (acc > best) best = acc;
        }
        s[p] = best;
    }
}

/* Ranking used by the selection: higher score first, equal scores by lower
 * page index; a NaN score ranks after every number. */
static _Thread_local const double *g_rank_scores;  /* per thread: callers may run units in parallel */
static int rank_cmp(const void *pa, const void *pb)
{
    int a = *(const int *)pa, b = *(const int *)pb;
    double sa = g_rank_scores[a], sb = g_rank_scores[b];
    int na = isnan(sa), nb = isnan(sb);
    if (na != nb) return na ? 1 : -1;
    if (!na && sa != sb) return sa > sb ? -1 : 1;
    return a < b ? -1 : (a > b ? 1 : 0);
}
static int int_cmp(const void *pa, const void *pb)
{
    int a = *(const int *)pa, b = *(const int *)pb;
    return a < b ? -1 : (a > b ? 1 : 0);
}

/* Pages kept for a budget of k pages, ascending logical ids, written to sel
 * (room for N ids).  Returns how many were kept:
 *   k >= N        -> all N pages;
 *   otherwise     -> the forced pages {0, N-1} plus the best k - |forced|
 *                    others (at least the forced pages, whatever k is). */
int oracle_select_pages(int N, const double *s, int k, int *sel)
{
    if (N <= 0) return 0;
    if (k >= N) {
        for (int p = 0; p < N; ++p) sel[p] = p;
        return N;
    }
    int nforced = N >= 2 ? 2 : 1;
    int take = k - nforced;
    if (take < 0) take = 0;
    int ncand = N - nforced;
    int *cand = (int *)malloc(sizeof(int) * (ncand > 0 ? ncand : 1));
    for (int i = 0; i < ncand; ++i) cand[i] = i + 1;  /* pages 1 .. N-2 */
    g_rank_scores = s;
    qsort(cand, (size_t)ncand, sizeof(int), rank_cmp);
    int n = 0;
    sel[n++] = 0;
    if (N >= 2) sel[n++] = N - 1;
    for (int i = 0; i < take && i < ncand; ++i) sel[n++] = cand[i];
    free(cand);
    qsort(sel, (size_t)n, sizeof(int), int_cmp);
    return n;
}

/* Masked softmax attention of G query heads over the tokens of the listed
 * pages with position < L.  out: [G][d].  Two passes (max, then exponentials)
 * as in the textbook definition.  An empty token set gives zeros. */
void oracle_attention(int G, int d, int L, int P, const double *q, const double *K,
                      const double *V, int npages, const int *pages, double scale,
                      double *out)
{
    for (int g = 0; g < G; ++g) {
        const double *qg = q + (size_t)g * d;
        double *og = out + (size_t)g * d;
        double m = -INFINITY;
        for (int i = 0; i < npages; ++i) {
            for (int t = pages[i] * P; t < (pages[i] + 1) * P && t < L; ++t) {
                double z = 0.0;
                for (int c = 0; c < d; ++c) z += qg[c] * K[(size_t)t * d + c];
                z *= scale;
                if (z > m) m = z;
            }
        }
        for (int c = 0; c < d; ++c) og[c] = 0.0;
        if (m == -INFINITY) continue;
        double denom = 0.0;
        for (int i = 0; i < npages; ++i) {
            for (int t = pages[i] * P; t < (pages[i] + 1) * P && t < L; ++t) {
                double z = 0.0;
                for (int c = 0; c < d; ++c) z += qg[c] * K[(size_t)t * d + c];
                double w = exp(z * scale - m);
                denom += w;
                for (int c = 0; c < d; ++c) og[c] += w * V[(size_t)t * d + c];
            }
        }
        for (int c = 0; c < d; ++c) og[c] /= denom;
    }
}

/* One decode step of one (sequence, KV head), from boxes already maintained:
 * score every page, keep the budget, attend over the kept pages.
 * sel must hold N ids; returns how many pages were kept. */
int oracle_decode_unit(int G, int d, int L, int P, const double *q, const double *K,
                       const double *V, const double *lo, const double *hi, int k,
                       double scale, double *scores, int *sel, double *out)
{
    int N = num_pages_of(L, P);
    if (N <= 0) {
        for (int i = 0; i < G * d; ++i) out[i] = 0.0;
        return 0;
    }
    oracle_page_scores(G, d, N, q, lo, hi, scores);
    int n = oracle_select_pages(N, scores, k, sel);
    oracle_attention(G, d, L, P, q, K, V, n, sel, scale, out);
    return n;
}

/* Share of the attention mass that falls on each page: the dense softmax
 * weights of each of the G query heads over all tokens below L, summed per
 * page and averaged over the heads.  mass: [N], sums to 1 when L > 0.  Used to
 * measure how well a page selection covers the true attention (the page hit
 * rate that the TinyServe abstract names beside cache reuse). */
void oracle_page_attention_mass(int G, int d, int L, int P, const double *q, const double *K,
                                double scale, double *mass)
{
    int N = num_pages_of(L, P);
    for (int p = 0; p < N; ++p) mass[p] = 0.0;
    if (L <= 0) return;
    double *z = (double *)malloc(sizeof(double) * (size_t)L);
    for (int g = 0; g < G; ++g) {
        const double *qg = q + (size_t)g * d;
        double m = -INFINITY;
        for (int t = 0; t < L; ++t) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += qg[c] * K[(size_t)t * d + c];
            z[t] = acc * scale;
            if (z[t] > m) m = z[t];
        }
        double denom = 0.0;
        for (int t = 0; t < L; ++t) denom += exp(z[t] - m);
        for (int t = 0; t < L; ++t) mass[t / P] += exp(z[t] - m) / denom / G;
    }
    free(z);
}

/* ------------------------------------------------------------------------
 * FP8 KV cache (e4m3 codes with a per-(page, KV head) scale).
 *
 * The TinyServe summary lists support for different KV formats among the
 * system's features without details; the readings here are: K and V are stored
 * as FP8 E4M3 codes (OCP 8-bit floating point, E4M3: 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits, subnormals, no infinities, S.1111.111 = NaN,
 * largest finite 448); every (page, KV head) keeps amax = the largest |x| of
 * the K (resp. V) values written into it, and scale s = amax / 448 (fp32); a
 * value x is stored as code(x / s); the page box holds the minimum and maximum
 * codes per channel (exact: every key of the page shares s).  When an append
 * raises a page's amax, the codes already in the page are re-quantized to the
 * new scale: code(dec(c) * s_old / s_new).  Those steps are fp32 operations
 * (each rounded to nearest), which this code performs in C float.
 * ---------------------------------------------------------------------- */

/* Value of an E4M3 code (NaN for S.1111.111). */
float oracle_e4m3_decode(unsigned char c)
{
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);                 /* subnormal: m * 2^-6 / 8 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return (float)(sign ? -v : v);
}

/* Nearest E4M3 code, ties to the even mantissa; finite values beyond 448
 * saturate to +-448; zero (of either sign) gives +0; NaN gives 0x7F. */
unsigned char oracle_e4m3_encode(float xf)
{
    double x = xf, a;
    int sign, e;
    double q, fl;
    long mant;
    if (x != x) return 0x7F;
    sign = x < 0;
    a = fabs(x);
    if (a > 448.0) return (unsigned char)((sign << 7) | 0x7E);
    if (a < ldexp(1.0, -6)) {                             /* subnormal range, step 2^-9 */
        q = a * 512.0;
        fl = floor(q);
        mant = (long)fl;
        if (q - fl > 0.5 || (q - fl == 0.5 && (mant & 1))) ++mant;
        if (mant == 0) return 0;                          /* +0 for both signs */
        if (mant == 8) return (unsigned char)((sign << 7) | (1 << 3));
        return (unsigned char)((sign << 7) | mant);
    }
    e = (int)floor(log2(a));
    if (ldexp(1.0, e) > a) --e;                           /* guard log2 rounding */
    if (ldexp(1.0, e + 1) <= a) ++e;
    q = (a / ldexp(1.0, e) - 1.0) * 8.0;                  /* exact: 0 <= q < 8 */
    fl = floor(q);
    mant = (long)fl;
    if (q - fl > 0.5 || (q - fl == 0.5 && (mant & 1))) ++mant;
    if (mant == 8) { mant = 0; ++e; }
    if (e > 8 || (e == 8 && mant > 6)) return (unsigned char)((sign << 7) | 0x7E);
    return (unsigned char)((sign << 7) | ((e + 7) << 3) | (int)mant);
}

/* Quantize one value with scale s (fp32); s == 0 stores 0. */
static unsigned char fp8_quant(float x, float s)
{
    if (s == 0.0f) return 0;
    return oracle_e4m3_encode(x / s);
}

/* Replay the quantized appends of ONE (sequence, KV head) tensor (K or V):
 * X [L][d] holds the input values (fp32), appended in chunks of chunk_lens
 * (summing to L).  Outputs: codes [L][d], amax [N], and per page the minimum
 * and maximum codes per channel lo, hi [N][d] (by value; compare the codes of
 * K, ignore for V). */
void oracle_fp8_append_replay(int L, int d, int P, const float *X, int nchunks, const int *chunk_lens,
                              unsigned char *codes, float *amax, unsigned char *lo, unsigned char *hi)
{
    int N = num_pages_of(L, P), t0 = 0;
    for (int p = 0; p < N; ++p) amax[p] = 0.0f;
    for (int k = 0; k < nchunks && t0 < L; ++k) {
        int t1 = t0 + chunk_lens[k];
        if (t1 > L) t1 = L;
        for (int p = t0 / P; p * P < t1; ++p) {
            int ts = t0 > p * P ? t0 : p * P;
            int te = t1 < (p + 1) * P ? t1 : (p + 1) * P;
            int fresh = (ts == p * P);
            float old = fresh ? 0.0f : amax[p], m = old;
            for (int t = ts; t < te; ++t)
                for (int c = 0; c < d; ++c) {
                    float v = fabsf(X[(size_t)t * d + c]);
                    if (v > m) m = v;
                }
            float s_old = old / 448.0f, s_new = m / 448.0f;
            if (!fresh && m > old)
                for (int t = p * P; t < ts; ++t)
                    for (int c = 0; c < d; ++c) {
                        unsigned char *cc = &codes[(size_t)t * d + c];
                        float x = oracle_e4m3_decode(*cc) * s_old;
                        *cc = fp8_quant(x, s_new);
                    }
            for (int t = ts; t < te; ++t)
                for (int c = 0; c < d; ++c)
                    codes[(size_t)t * d + c] = fp8_quant(X[(size_t)t * d + c], s_new);
            amax[p] = m;
            for (int c = 0; c < d; ++c) {
                unsigned char mn = codes[(size_t)(p * P) * d + c], mx = mn;
                for (int t = p * P + 1; t < te; ++t) {
                    unsigned char v = codes[(size_t)t * d + c];
                    if (oracle_e4m3_decode(v) < oracle_e4m3_decode(mn)) mn = v;
                    if (oracle_e4m3_decode(v) > oracle_e4m3_decode(mx)) mx = v;
                }
                lo[(size_t)p * d + c] = mn;
                hi[(size_t)p * d + c] = mx;
            }
        }
        t0 = t1;
    }
}
