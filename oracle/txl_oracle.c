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
 * Readings where the pages leave a step open:
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
 *   lse    : [B][H][L]         (optional, may be NULL: each row's log of its
 *                               softmax denominator)
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
 * doubles.  The exact definition: no blocking, no online rescaling.  When
 * lse_out is not NULL it receives the natural log of the softmax denominator,
 * log sum_j exp(s_j) over the visible keys. */
static void one_row(const double *q, const double *k, const double *v,
                    const double *r, const double *u, const double *w,
                    long B, long H, long D, long L, long M, long b, long h,
                    long i, double *s, double *out_row, double *prob_row,
                    double *lse_out)
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
    if (lse_out) *lse_out = mx + log(z);
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
                         double *out, double *prob, double *lse, int nthreads)
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
                one_row(q, k, v, r, u, w, B, H, D, L, M, b, h, i, s, row, prow,
                        lse ? lse + (b * H + h) * L + i : NULL);
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
                    out_rows + x * D, NULL, NULL);
        }
        free(s);
    }
}

/* Gradients of one layer call for a given output gradient dout (the
 * backward of the function above, written out by the chain rule).  For one
 * query row (b, h, i), with P_j the softmax weights and A_j the unscaled
 * four-term score:
 *   dP_j  = dout_i . v_j
 *   dS_j  = P_j (dP_j - sum_l P_l dP_l)          (softmax, on the scaled score)
 *   dA_j  = dS_j / sqrt(D)
 *   dq_i += dA_j (k_j + r_{T-1-off})             (both bias-shifted queries)
 *   dk_j += dA_j (q_i + u)      dv_j += P_j dout_i
 *   dr_{T-1-off} += dA_j (q_i + v)               (summed over the batch)
 *   du   += dA_j k_j            dw   += dA_j r_{T-1-off}
 * with off = M+i-j the relative distance of the visible pair (j <= M+i).
 * Every input gets its gradient, the memory rows of k and v included: the
 * stop-gradient of Section 3.2 stops at the cached hidden states, not at the
 * keys and values computed from them.  dr_part, du_part, dw_part are scratch
 * of B*H*T*D, B*H*D, B*H*D doubles (one slice per (b, h), summed at the end
 * so that the parallel loop shares no accumulator). */
void txl_oracle_rel_attn_bwd(const double *q, const double *k, const double *v,
                             const double *r, const double *u, const double *w,
                             const double *dout, long B, long H, long D, long L,
                             long M, double *dq, double *dk, double *dv, double *dr,
                             double *du, double *dw, double *dr_part,
                             double *du_part, double *dw_part, int nthreads)
{
    const long T = M + L;
    const long nbh = B * H;
    const double scale = 1.0 / sqrt((double)D);
    for (long x = 0; x < L * B * H * D; ++x) dq[x] = 0.0;
    for (long x = 0; x < T * B * H * D; ++x) dk[x] = dv[x] = 0.0;
    for (long x = 0; x < nbh * T * D; ++x) dr_part[x] = 0.0;
    for (long x = 0; x < nbh * D; ++x) du_part[x] = dw_part[x] = 0.0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (long bh = 0; bh < nbh; ++bh) {
            const long b = bh / H, h = bh % H;
            const double *uh = u + h * D, *wh = w + h * D;
            double *drp = dr_part + bh * T * D, *dup = du_part + bh * D, *dwp = dw_part + bh * D;
            for (long i = 0; i < L; ++i) {
                const double *qi = q + ((i * B + b) * H + h) * D;
                const double *gi = dout + ((i * B + b) * H + h) * D;
                double *dqi = dq + ((i * B + b) * H + h) * D;
                const long last = M + i;
                double mx = -INFINITY;
                for (long j = 0; j <= last; ++j) {
                    const long off = M + i - j;
                    const double *rr = r + ((T - 1 - off) * H + h) * D;
                    const double *kj = k + ((j * B + b) * H + h) * D;
                    double a = 0.0;
                    for (long d = 0; d < D; ++d) a += (qi[d] + uh[d]) * kj[d] + (qi[d] + wh[d]) * rr[d];
                    s[j] = a * scale;
                    if (s[j] > mx) mx = s[j];
                }
                double z = 0.0;
                for (long j = 0; j <= last; ++j) {
                    s[j] = exp(s[j] - mx);
                    z += s[j];
                }
                double delta = 0.0;
                for (long j = 0; j <= last; ++j) {
                    s[j] /= z; /* P_j */
                    const double *vj = v + ((j * B + b) * H + h) * D;
                    double g = 0.0;
                    for (long d = 0; d < D; ++d) g += gi[d] * vj[d];
                    dp[j] = g;
                    delta += s[j] * g;
                }
                for (long j = 0; j <= last; ++j) {
                    const long off = M + i - j;
                    const long t = T - 1 - off;
                    const double *rr = r + (t * H + h) * D;
                    const double *kj = k + ((j * B + b) * H + h) * D;
                    double *dkj = dk + ((j * B + b) * H + h) * D;
                    double *dvj = dv + ((j * B + b) * H + h) * D;
                    const double da = s[j] * (dp[j] - delta) * scale;
                    for (long d = 0; d < D; ++d) {
                        dqi[d] += da * (kj[d] + rr[d]);
                        dkj[d] += da * (qi[d] + uh[d]);
                        dvj[d] += s[j] * gi[d];
                        drp[t * D + d] += da * (qi[d] + wh[d]);
                        dup[d] += da * kj[d];
                        dwp[d] += da * rr[d];
                    }
                }
            }
        }
        free(s);
        free(dp);
    }
    for (long x = 0; x < T * H * D; ++x) dr[x] = 0.0;
    for (long x = 0; x < H * D; ++x) du[x] = dw[x] = 0.0;
    for (long bh = 0; bh < nbh; ++bh) {
        const long h = bh % H;
        for (long t = 0; t < T; ++t)
            for (long d = 0; d < D; ++d) dr[(t * H + h) * D + d] += dr_part[(bh * T + t) * D + d];
        for (long d = 0; d < D; ++d) {
            du[h * D + d] += du_part[bh * D + d];
            dw[h * D + d] += dw_part[bh * D + d];
        }
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
