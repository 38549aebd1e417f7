/*
 * sdpa_oracle.c -- float64 CPU oracle for the scaled-dot-product attention forward pass.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke() and
 * bench.py's cpu_baseline / reference leg may load this library.  The CUDA path never
 * links, includes or calls anything in this directory, and this file includes nothing
 * from the CUDA path.
 *
 * What is computed, and where it is defined:
 *   "An Optimal Mapper Meets a Real GPU" (tinglin.vercel.app), sections "Ground rules"
 *   and "Experiment one" (the Cases table): scaled-dot-product attention with FP16
 *   inputs, query length equal to key/value length, with or without a causal mask,
 *   gated against PyTorch SDPA.  Its three stages are QK (scores), softmax (row max,
 *   exp, sum, divide; see item (3) of the missing cost terms in "Experiment one") and
 *   AV (weights times values).
 *   "STAGE_D.md" of nvfp4-megamoe-kernel, section 4 ("Guard Dead Code with const_expr"):
 *   the attention kernel also yields the row log-sum-exp (LSE) of the scaled logits.
 *   Same page, section 2 ("External k_sub Merge is Mathematically Impossible"):
 *   head_dim sub-tiles add up in logit space, S = S_0 + S_1, before the softmax.
 *
 * The definition written out, for every (b, h, i), in float64 from the exact fp16
 * input values (the caller converts fp16 -> float64, which is exact):
 *     s_j  = scale * sum_{t=0}^{d-1} q[b,h,i,t] * k[b,h,j,t]        j < L (causal: j <= i)
 *     m    = max_j s_j,   e_j = exp(s_j - m),   l = sum_j e_j
 *     O[b,h,i,c] = (sum_j e_j * v[b,h,j,c]) / l
 *     LSE[b,h,i] = m + log(l)                                          (natural log)
 * No blocking, no online softmax, no split of d: the sum over t runs in ascending
 * order and every intermediate is float64.  Every buffer is heap-allocated (large
 * per-thread stack buffers are avoided on purpose).
 *
 * Layout of every tensor: [B, H, L, d] (or [B, H, L, L] for scores), contiguous, the
 * layout of PyTorch's scaled_dot_product_attention, which the first page gates against.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One output row (b, h, i) of the forward pass, straight from the definition above.
 * `srow` is caller-owned scratch of at least L doubles. */
static void sdpa_row(const double *q, const double *k, const double *v, double *o_row,
                     double *lse_out, long L, long d, int causal, double scale,
                     long bh, long i, double *srow)
{
    const double *qi = q + (bh * L + i) * d;
    const double *kh = k + bh * L * d;
    const double *vh = v + bh * L * d;
    long jmax = causal ? i + 1 : L; /* keys j <= i under the causal mask */

    /* scores */
    for (long j = 0; j < jmax; ++j) {
        const double *kj = kh + j * d;
        double acc = 0.0;
        for (long t = 0; t < d; ++t)
            acc += qi[t] * kj[t];
        srow[j] = scale * acc;
    }
    /* softmax: max, exp, sum */
    double m = -INFINITY;
    for (long j = 0; j < jmax; ++j)
        if (srow[j] > m)
            m = srow[j];
    double l = 0.0;
    for (long j = 0; j < jmax; ++j) {
        srow[j] = exp(srow[j] - m);
        l += srow[j];
    }
    /* weights times values, then divide */
    for (long c = 0; c < d; ++c) {
        double acc = 0.0;
        for (long j = 0; j < jmax; ++j)
            acc += srow[j] * vh[j * d + c];
        o_row[c] = acc / l;
    }
    *lse_out = m + log(l);
}

static int resolve_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Full forward pass.  o: [B,H,L,d], lse: [B,H,L].  Rows are independent, so they are
 * spread over `nthreads` OpenMP threads (0 = all available); the arithmetic of a row
 * does not depend on the thread count.  Returns the thread count used, or -1 if the
 * scratch allocation failed. */
int oracle_sdpa_fwd(const double *q, const double *k, const double *v, double *o,
                    double *lse, int B, int H, int L, int d, int causal, double scale,
                    int nthreads)
{
    int nt = resolve_threads(nthreads);
    long nrows = (long)B * H * L;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)nt * (size_t)(L > 0 ? L : 1));
    if (!scratch)
        return -1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 16)
    for (long r = 0; r < nrows; ++r) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        long bh = r / L, i = r % L;
        sdpa_row(q, k, v, o + r * d, lse + r, L, d, causal, scale, bh, i,
                 scratch + (size_t)tid * (size_t)L);
    }
    free(scratch);
    return nt;
}

/* The same rows as oracle_sdpa_fwd, but only for the flat row indices listed in `rows`
 * (row = (b*H + h)*L + i).  o: [nrows, d], lse: [nrows].  Used to check a sample of the
 * outputs of a problem too large to recompute in full. */
int oracle_sdpa_fwd_rows(const double *q, const double *k, const double *v, double *o,
                         double *lse, int B, int H, int L, int d, int causal,
                         double scale, const int64_t *rows, long nrows, int nthreads)
{
    int nt = resolve_threads(nthreads);
    long total = (long)B * H * L;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)nt * (size_t)(L > 0 ? L : 1));
    if (!scratch)
        return -1;
    int bad = 0;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 4) reduction(| : bad)
    for (long n = 0; n < nrows; ++n) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        long r = (long)rows[n];
        if (r < 0 || r >= total) {
            bad = 1;
            continue;
        }
        long bh = r / L, i = r % L;
        sdpa_row(q, k, v, o + n * d, lse + n, L, d, causal, scale, bh, i,
                 scratch + (size_t)tid * (size_t)L);
    }
    free(scratch);
    return bad ? -2 : nt;
}

/* Stage 1 alone (QK): s[b,h,i,j] = scale * sum_{t=t0}^{t1-1} q[b,h,i,t] * k[b,h,j,t]
 * for every i, j (no mask).  With [t0, t1) a part of [0, d) this is one head_dim
 * sub-tile's share of the logits. */
void oracle_scores(const double *q, const double *k, double *s, int B, int H, int L,
                   int d, double scale, int t0, int t1)
{
    long nbh = (long)B * H;
#pragma omp parallel for schedule(static)
    for (long bh = 0; bh < nbh; ++bh)
        for (long i = 0; i < L; ++i) {
            const double *qi = q + (bh * L + i) * d;
            for (long j = 0; j < L; ++j) {
                const double *kj = k + (bh * L + j) * d;
                double acc = 0.0;
                for (long t = t0; t < t1; ++t)
                    acc += qi[t] * kj[t];
                s[(bh * L + i) * L + j] = scale * acc;
            }
        }
}

/* Stage 2 alone (softmax) on given logits s [B,H,L,L]: p[b,h,i,j] is the masked row
 * softmax (0 where the causal mask removes j > i) and lse[b,h,i] its log-sum-exp. */
void oracle_softmax(const double *s, double *p, double *lse, int B, int H, int L,
                    int causal)
{
    long nrows = (long)B * H * L;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < nrows; ++r) {
        long i = r % L;
        long jmax = causal ? i + 1 : L;
        const double *sr = s + r * L;
        double *pr = p + r * L;
        double m = -INFINITY;
        for (long j = 0; j < jmax; ++j)
            if (sr[j] > m)
                m = sr[j];
        double l = 0.0;
        for (long j = 0; j < jmax; ++j) {
            pr[j] = exp(sr[j] - m);
            l += pr[j];
        }
        for (long j = 0; j < jmax; ++j)
            pr[j] /= l;
        for (long j = jmax; j < L; ++j)
            pr[j] = 0.0;
        lse[r] = m + log(l);
    }
}

/* Stage 3 alone (AV): o[b,h,i,c] = sum_j p[b,h,i,j] * v[b,h,j,c]. */
void oracle_pv(const double *p, const double *v, double *o, int B, int H, int L, int d)
{
    long nbh = (long)B * H;
#pragma omp parallel for schedule(static)
    for (long bh = 0; bh < nbh; ++bh)
        for (long i = 0; i < L; ++i) {
            const double *pr = p + (bh * L + i) * L;
            for (long c = 0; c < d; ++c) {
                double acc = 0.0;
                for (long j = 0; j < L; ++j)
                    acc += pr[j] * v[(bh * L + j) * d + c];
                o[(bh * L + i) * d + c] = acc;
            }
        }
}
