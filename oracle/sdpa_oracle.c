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
 *
 * Backward ("Validating Memory-Optimal Transformer Kernels on Real Hardware", section 4,
 * "Paper II: Backward Pass and Fused Forward+Backward": the gradients GQ, GK, GV of the
 * attention output, through the gradient GS of the scores) is the derivative of the same
 * definition for a given upstream gradient dO; see oracle_sdpa_bwd.
 *
 * Decode ("Validating Memory-Optimal Transformer Kernels on Real Hardware", section 5,
 * "Paper III: Inference (Decode)": one new token per sequence attends to the whole cached
 * sequence, at O(n) cost in the sequence length n) is the same definition with a single
 * query row per (b, h) and every one of the L keys visible; see oracle_decode_f16.
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

/* IEEE 754 binary16 -> double, from the format's definition: 1 sign bit, 5 exponent bits
 * (bias 15), 10 fraction bits.  Exponent 0: zero or subnormal, fraction * 2^-24;
 * exponent 31: infinity (fraction 0) or NaN; otherwise (1024 + fraction) * 2^(e - 25).
 * Exact: every binary16 value is a double. */
static double f16_to_f64(uint16_t h)
{
    int e = (h >> 10) & 31, f = h & 1023;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(f + 1024), e - 25);
    return (h >> 15) ? -mag : mag;
}

/* The conversion above over an array (exported so that it can be checked on its own). */
void oracle_f16_to_f64(const uint16_t *h, double *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = f16_to_f64(h[i]);
}

/* Decode: one query row per head bh against all L keys of that head, no mask.
 * Inputs are raw fp16 bits, q [BH, d] and k, v [BH, L, d], converted element by element
 * (the full key and value sets of a long sequence are never copied to float64).  For
 * every head listed in `heads` (n_heads of them; NULL: all BH heads, in order):
 *     s_j = scale * sum_{t=0}^{d-1} q[bh,t] * k[bh,j,t]        j < L
 *     m = max_j s_j,   e_j = exp(s_j - m),   l = sum_j e_j
 *     o[n, c] = (sum_j e_j * v[bh,j,c]) / l,   lse[n] = m + log(l)
 * with n the position of bh in the list; float64 throughout, sums in ascending order.
 * Returns the thread count used, -1 if scratch allocation failed, -2 for a head index out
 * of range. */
int oracle_decode_f16(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *o,
                      double *lse, long BH, long L, int d, double scale, const int64_t *heads,
                      long n_heads, int nthreads)
{
    int nt = resolve_threads(nthreads);
    long n = heads ? n_heads : BH;
    size_t per = (size_t)(L > 0 ? L : 1) + (size_t)d + (size_t)d;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)nt * per);
    if (!scratch)
        return -1;
    int bad = 0;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1) reduction(| : bad)
    for (long i = 0; i < n; ++i) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        long bh = heads ? (long)heads[i] : i;
        if (bh < 0 || bh >= BH) {
            bad = 1;
            continue;
        }
        double *srow = scratch + (size_t)tid * per;
        double *qf = srow + (L > 0 ? L : 1);
        double *acc = qf + d;
        for (int t = 0; t < d; ++t)
            qf[t] = f16_to_f64(q[bh * d + t]);
        /* scores */
        for (long j = 0; j < L; ++j) {
            const uint16_t *kj = k + ((size_t)bh * L + j) * d;
            double dot = 0.0;
            for (int t = 0; t < d; ++t)
                dot += qf[t] * f16_to_f64(kj[t]);
            srow[j] = scale * dot;
        }
        /* softmax: max, exp, sum */
        double m = -INFINITY;
        for (long j = 0; j < L; ++j)
            if (srow[j] > m)
                m = srow[j];
        double l = 0.0;
        for (long j = 0; j < L; ++j) {
            srow[j] = exp(srow[j] - m);
            l += srow[j];
        }
        /* weights times values (key order ascending for every column), then divide */
        for (int c = 0; c < d; ++c)
            acc[c] = 0.0;
        for (long j = 0; j < L; ++j) {
            const uint16_t *vj = v + ((size_t)bh * L + j) * d;
            for (int c = 0; c < d; ++c)
                acc[c] += srow[j] * f16_to_f64(vj[c]);
        }
        for (int c = 0; c < d; ++c)
            o[i * d + c] = acc[c] / l;
        lse[i] = m + log(l);
    }
    free(scratch);
    return bad ? -2 : nt;
}

/* Backward pass of the forward definition above: for an upstream gradient dO of O
 * (every tensor [B, H, L, d], float64), per head, with S, P the scaled masked logits and
 * their row softmax:
 *     dV = P^T dO
 *     dP = dO V^T
 *     dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)        (the softmax's Jacobian; 0 where masked)
 *     dQ = scale * dS K,      dK = scale * dS^T Q
 * Straight from the definition: the full L x L matrices of one head are formed (heap
 * buffers), sums in ascending index order.  Heads are spread over `nthreads` threads.
 * Returns the thread count used, or -1 if scratch allocation failed. */
int oracle_sdpa_bwd(const double *q, const double *k, const double *v, const double *dout, double *dq,
                    double *dk, double *dv, int B, int H, int L, int d, int causal, double scale, int nthreads)
{
    int nt = resolve_threads(nthreads);
    long nbh = (long)B * H;
    size_t ll = (size_t)L * (size_t)L;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)nt * 2 * (ll > 0 ? ll : 1));
    if (!scratch)
        return -1;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (long bh = 0; bh < nbh; ++bh) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *P = scratch + (size_t)tid * 2 * ll;
        double *dS = P + ll;
        const double *qh = q + bh * L * d, *kh = k + bh * L * d, *vh = v + bh * L * d, *doh = dout + bh * L * d;
        double *dqh = dq + bh * L * d, *dkh = dk + bh * L * d, *dvh = dv + bh * L * d;
        /* P: row softmax of the scaled, masked logits (masked entries 0) */
        for (long i = 0; i < L; ++i) {
            long jmax = causal ? i + 1 : L;
            double m = -INFINITY;
            for (long j = 0; j < jmax; ++j) {
                double acc = 0.0;
                for (long t = 0; t < d; ++t)
                    acc += qh[i * d + t] * kh[j * d + t];
                P[i * L + j] = scale * acc;
                if (P[i * L + j] > m)
                    m = P[i * L + j];
            }
            double l = 0.0;
            for (long j = 0; j < jmax; ++j) {
                P[i * L + j] = exp(P[i * L + j] - m);
                l += P[i * L + j];
            }
            for (long j = 0; j < jmax; ++j)
                P[i * L + j] /= l;
            for (long j = jmax; j < L; ++j)
                P[i * L + j] = 0.0;
        }
        /* dP = dO V^T and dS = P (dP - rowsum(P dP)) */
        for (long i = 0; i < L; ++i) {
            long jmax = causal ? i + 1 : L;
            double rs = 0.0;
            for (long j = 0; j < jmax; ++j) {
                double acc = 0.0;
                for (long t = 0; t < d; ++t)
                    acc += doh[i * d + t] * vh[j * d + t];
                dS[i * L + j] = acc;
                rs += P[i * L + j] * acc;
            }
            for (long j = 0; j < jmax; ++j)
                dS[i * L + j] = P[i * L + j] * (dS[i * L + j] - rs);
            for (long j = jmax; j < L; ++j)
                dS[i * L + j] = 0.0;
        }
        /* dV = P^T dO,  dK = scale dS^T Q */
        for (long j = 0; j < L; ++j)
            for (long t = 0; t < d; ++t) {
                double av = 0.0, ak = 0.0;
                for (long i = 0; i < L; ++i) {
                    av += P[i * L + j] * doh[i * d + t];
                    ak += dS[i * L + j] * qh[i * d + t];
                }
                dvh[j * d + t] = av;
                dkh[j * d + t] = scale * ak;
            }
        /* dQ = scale dS K */
        for (long i = 0; i < L; ++i)
            for (long t = 0; t < d; ++t) {
                double aq = 0.0;
                for (long j = 0; j < L; ++j)
                    aq += dS[i * L + j] * kh[j * d + t];
                dqh[i * d + t] = scale * aq;
            }
    }
    free(scratch);
    return nt;
}
