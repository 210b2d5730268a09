/*
 * txl_oracle.c -- plain, slow, float64 CPU reference for Transformer-XL
 * segment-level relative multi-head attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg load this library.  The product path (the
 * CUDA library behind include/txl.h) never links, loads or calls it, and this
 * file includes nothing from that library.
 *
 * What it computes follows "Transformer-XL: Attentive Language Models Beyond a
 * Fixed-Length Context" (Dai et al., 2019):
 *   - Section 3.3, the per-layer computing procedure: the score of query i
 *     against key j is
 *         A_ij = q_i.k_j + q_i.(W_kR R_{i-j}) + u.k_j + v.(W_kR R_{i-j})
 *     (terms a, b, c, d), and the attention output is the masked softmax of A
 *     times the values.
 *   - Section 3.2: keys and values cover the extended context
 *     [memory (M rows, oldest first); current segment (L rows)].
 *   - Appendix B: the relative distance of a visible pair lies in 0..M+L-1 and
 *     the projected table is stored reversed, Q_k = W_kR R_{M+L-1-k}; the
 *     query at segment position i sees key j exactly when j <= M+i.
 * Readings where the pages leave a step open (all listed in the design doc):
 *   - the whole score A is scaled by 1/sqrt(d_head) before the softmax (the
 *     scaled softmax of the vanilla attention on the summary page);
 *   - heads are independent, u and v are per head, and the projected table r
 *     is shared by every sequence of the batch.
 *
 * Layouts (all row-major, T = M + L):
 *   q, out : [L][B][H][D]      k, v : [T][B][H][D]
 *   r      : [T][H][D], row t holds W_kR R_{T-1-t}
 *   u, w   : [H][D]            (w is the paper's v bias)
 *   prob   : [B][H][L][T]      (optional, may be NULL)
 *
 * Status: parity pinned.  The pins (tests/test_oracle_pins.py) check this code
 * against the four-term expansion from hidden states, the Appendix B
 * left-shift route, an absolute-position sinusoid route, the textbook softmax
 * attention of a library routine and the segment-recurrence identity.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One query row (b, h, i): the masked, scaled softmax over keys 0..M+i of the
 * four-term score, then the weighted sum of the values.  s is scratch of T
 * doubles.  The exact definition: no blocking, no online rescaling. */
static void one_row(const double *q, const double *k, const double *v,
                    const double *r, const double *u, const double *w,
                    long B, long H, long D, long L, long M, long b, long h,
                    long i, double *s, double *out_row, double *prob_row)
{
    const long T = M + L;
    const double scale = 1.0 / sqrt((double)D);
    const double *qi = q + ((i * B + b) * H + h) * D;
    const double *uh = u + h * D;
    const double *wh = w + h * D;
    const long last = M + i; /* the last visible key (Appendix B zero pattern) */
    double mx = -INFINITY;

    for (long j = 0; j <= last; ++j) {
        const long off = M + i - j;                      /* relative distance i-j */
        const double *rr = r + ((T - 1 - off) * H + h) * D; /* Q_{T-1-off} = W_kR R_off */
        const double *kj = k + ((j * B + b) * H + h) * D;
        double a = 0.0;
        for (long d = 0; d < D; ++d) {
            /* terms (a)+(c): (q_i + u).k_j ; terms (b)+(d): (q_i + v).r */
            a += (qi[d] + uh[d]) * kj[d] + (qi[d] + wh[d]) * rr[d];
        }
        s[j] = a * scale;
        if (s[j] > mx) mx = s[j];
    }
    double z = 0.0;
    for (long j = 0; j <= last; ++j) {
        s[j] = exp(s[j] - mx);
        z += s[j];
    }
    for (long j = 0; j <= last; ++j) s[j] /= z;
    for (long d = 0; d < D; ++d) {
        double o = 0.0;
        for (long j = 0; j <= last; ++j) o += s[j] * v[((j * B + b) * H + h) * D + d];
        out_row[d] = o;
    }
    if (prob_row) {
        for (long j = 0; j < T; ++j) prob_row[j] = (j <= last) ? s[j] : 0.0;
    }
}

/* Full layer call: every (b, h, i).  OpenMP over (b, h) when nthreads > 0. */
void txl_oracle_rel_attn(const double *q, const double *k, const double *v,
                         const double *r, const double *u, const double *w,
                         long B, long H, long D, long L, long M,
                         double *out, double *prob, int nthreads)
{
    const long T = M + L;
    const long nbh = B * H;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double *row = (double *)malloc(sizeof(double) * (size_t)(D > 0 ? D : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (long bh = 0; bh < nbh; ++bh) {
            const long b = bh / H, h = bh % H;
            for (long i = 0; i < L; ++i) {
                double *prow = prob ? prob + ((b * H + h) * L + i) * T : NULL;
                one_row(q, k, v, r, u, w, B, H, D, L, M, b, h, i, s, row, prow);
                double *o = out + ((i * B + b) * H + h) * D;
                for (long d = 0; d < D; ++d) o[d] = row[d];
            }
        }
        free(s);
        free(row);
    }
}

/* Selected rows only: rows holds n triples (b, h, i); out_rows is [n][D].
 * Used to check full-size launches on a sample of their outputs. */
void txl_oracle_rel_attn_rows(const double *q, const double *k, const double *v,
                              const double *r, const double *u, const double *w,
                              long B, long H, long D, long L, long M,
                              const int64_t *rows, long n, double *out_rows,
                              int nthreads)
{
    const long T = M + L;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (long x = 0; x < n; ++x) {
            one_row(q, k, v, r, u, w, B, H, D, L, M, (long)rows[3 * x],
                    (long)rows[3 * x + 1], (long)rows[3 * x + 2], s,
                    out_rows + x * D, NULL);
        }
        free(s);
    }
}

/* Number of threads OpenMP would use (1 when built without OpenMP). */
int txl_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
