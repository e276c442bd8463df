/*
 * Oracle for exact softmax attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load this library.  The product path (the CUDA library) never
 * calls it, links it or shares a header with it.
 *
 * What it computes is the plain definition of scaled dot-product attention
 * as the pages state it:
 *   - "Triton Ascend Attention" (skillmd.com), section "标准 Attention 计算流程":
 *     Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V, done in three stages
 *     (scores, row softmax, weighted sum), with the score matrix materialised.
 *   - "FlashAttention-2 forward in Triton" (wsisp.com), the passage stating that
 *     FlashAttention computes exactly S = Q K^T, P = softmax(S), O = P V, and the
 *     epilogue of the outer kernel, where the stored per-row statistic is
 *     m + log(l) (the log-sum-exp of the scaled scores, natural log).
 *   - Causal masking keeps key j for query i iff i >= j ("flash-attention-kernel"
 *     skill card, the note "offs_m >= offs_n not offs_m > offs_n"), i.e. the
 *     diagonal is kept and rows/keys are aligned at index 0.
 *
 * Every value is double precision.  Per query row the oracle materialises the
 * full score row S[i, :] and probability row P[i, :] (length Lk), then forms
 * O[i, :] = sum_j P[i, j] V[j, :] in index order.  There is no tiling, no online
 * recurrence and no reordering beyond what the definition states.
 *
 * Readings where the pages are silent (each is restated in the design notes):
 *   - keys j >= Lk do not exist (no phantom zero-score keys);
 *   - the scale multiplies the raw dot product before the max and the exp;
 *   - masked pairs are excluded (weight exactly 0), not given a finite penalty;
 *   - causal alignment for Lq != Lk is top-left: key j allowed iff j <= i.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Return codes. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

/* Number of keys query row i may attend to (a prefix 0..n-1 of the keys). */
static long allowed_keys(long i, long Lk, int causal)
{
    if (!causal) return Lk;
    return (i + 1 < Lk) ? (i + 1) : Lk;
}

/* One query row of one head, straight from the definition.
 * q: [D]; K, V: [Lk, D] row-major; S, P: caller scratch of length Lk.
 * Writes o[D], *lse, and (if p_out) the probability row p_out[Lk] with zeros
 * at masked keys. */
static void attend_row(const double *q, const double *K, const double *V,
                       long Lk, long D, long n_allowed, double scale,
                       double *S, double *P, double *o, double *lse, double *p_out)
{
    /* Stage 1: scores S_ij = scale * <q_i, k_j> over the allowed keys. */
    for (long j = 0; j < n_allowed; ++j) {
        double dot = 0.0;
        for (long d = 0; d < D; ++d) dot += q[d] * K[j * D + d];
        S[j] = scale * dot;
    }
    /* Stage 2: row softmax, stabilised by the row maximum. */
    double m = -INFINITY;
    for (long j = 0; j < n_allowed; ++j)
        if (S[j] > m) m = S[j];
    double l = 0.0;
    for (long j = 0; j < n_allowed; ++j) {
        P[j] = exp(S[j] - m);
        l += P[j];
    }
    for (long j = 0; j < n_allowed; ++j) P[j] /= l;
    /* Stage 3: weighted sum of value rows. */
    for (long d = 0; d < D; ++d) o[d] = 0.0;
    for (long j = 0; j < n_allowed; ++j) {
        const double w = P[j];
        for (long d = 0; d < D; ++d) o[d] += w * V[j * D + d];
    }
    /* Log-sum-exp of the scaled scores over the allowed keys: m + ln(l). */
    *lse = m + log(l);
    if (p_out) {
        for (long j = 0; j < n_allowed; ++j) p_out[j] = P[j];
        for (long j = n_allowed; j < Lk; ++j) p_out[j] = 0.0;
    }
}

/*
 * Attention for one (batch, head) slice, on a chosen set of query rows.
 *   Q: [Lq, D], K: [Lk, D], V: [Lk, D], all row-major doubles.
 *   rows: nrows query indices in [0, Lq); NULL means all rows 0..Lq-1
 *         (then nrows must equal Lq).
 *   O: [nrows, D] out; LSE: [nrows] out; P: [nrows, Lk] out or NULL.
 *   nthreads: OpenMP threads to use (<= 0: the runtime default).
 * Returns ORACLE_OK, or an error code (argument errors before any output is written;
 * ORACLE_NO_MEMORY with the outputs incomplete).
 */
int oracle_attn_head(const double *Q, const double *K, const double *V,
                     long Lq, long Lk, long D, int causal, double scale,
                     const long *rows, long nrows,
                     double *O, double *LSE, double *P, int nthreads)
{
    if (!Q || !K || !V || !O || !LSE) return ORACLE_BAD_ARG;
    if (Lq < 0 || Lk < 1 || D < 1 || nrows < 0) return ORACLE_BAD_ARG;
    if (!rows && nrows != Lq) return ORACLE_BAD_ARG;
    if (rows)
        for (long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= Lq) return ORACLE_BAD_ARG;
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)Lk);
        double *Pr = (double *)malloc(sizeof(double) * (size_t)Lk);
        const int have = S && Pr;
        if (!have) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_NO_MEMORY;
        }
        /* Every thread of the team meets the worksharing loop; one without its row
         * buffers takes its share of rows and skips them (the call then fails). */
        {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (long r = 0; r < nrows; ++r) {
                if (!have) continue;
                const long i = rows ? rows[r] : r;
                attend_row(Q + i * D, K, V, Lk, D, allowed_keys(i, Lk, causal), scale,
                           S, Pr, O + r * D, LSE + r, P ? P + r * Lk : NULL);
            }
        }
        free(S);
        free(Pr);
    }
    return status;
}

/*
 * Whole-tensor attention over contiguous [B, H, L, D] doubles:
 *   O: [B, H, Lq, D], LSE: [B, H, Lq], P: [B, H, Lq, Lk] or NULL.
 */
int oracle_attn_full(const double *Q, const double *K, const double *V,
                     long B, long H, long Lq, long Lk, long D, int causal, double scale,
                     double *O, double *LSE, double *P, int nthreads)
{
    if (B < 0 || H < 0) return ORACLE_BAD_ARG;
    for (long bh = 0; bh < B * H; ++bh) {
        int rc = oracle_attn_head(Q + bh * Lq * D, K + bh * Lk * D, V + bh * Lk * D,
                                  Lq, Lk, D, causal, scale, NULL, Lq,
                                  O + bh * Lq * D, LSE + bh * Lq,
                                  P ? P + bh * Lq * Lk : NULL, nthreads);
        if (rc != ORACLE_OK) return rc;
    }
    return ORACLE_OK;
}


/*
 * Local (sliding-window) attention for one (batch, head) slice: query row i may
 * attend to key j iff  i - left <= j <= i + right  and 0 <= j < Lk, where left or
 * right = -1 means unbounded on that side ("FlashAttention-2 forward in Triton",
 * wsisp.com: local / sliding-window attention, whose queries do not attend to all
 * tokens).  Rows and keys are aligned at index 0 as in the causal case, which is
 * left = -1, right = 0.  The allowed keys of a row form one contiguous range, so
 * each row is the definition above applied to that range of K and V rows.
 * A row with no allowed key is an argument error (ORACLE_BAD_ARG).
 * Arguments as oracle_attn_head; P (if given) is zero outside the range.
 */
int oracle_attn_head_window(const double *Q, const double *K, const double *V,
                            long Lq, long Lk, long D, long left, long right, double scale,
                            const long *rows, long nrows,
                            double *O, double *LSE, double *P, int nthreads)
{
    if (!Q || !K || !V || !O || !LSE) return ORACLE_BAD_ARG;
    if (Lq < 0 || Lk < 1 || D < 1 || nrows < 0 || left < -1 || right < -1) return ORACLE_BAD_ARG;
    if (!rows && nrows != Lq) return ORACLE_BAD_ARG;
    for (long r = 0; r < nrows; ++r) {
        const long i = rows ? rows[r] : r;
        if (i < 0 || i >= Lq) return ORACLE_BAD_ARG;
        const long lo = (left < 0 || i - left < 0) ? 0 : i - left;
        const long hi = (right < 0 || i + right > Lk - 1) ? Lk - 1 : i + right;
        if (lo > hi) return ORACLE_BAD_ARG;
    }
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)Lk);
        double *Pr = (double *)malloc(sizeof(double) * (size_t)Lk);
        const int have = S && Pr;
        if (!have) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_NO_MEMORY;
        }
        /* Every thread of the team meets the worksharing loop; one without its row
         * buffers takes its share of rows and skips them (the call then fails). */
        {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (long r = 0; r < nrows; ++r) {
                if (!have) continue;
                const long i = rows ? rows[r] : r;
                const long lo = (left < 0 || i - left < 0) ? 0 : i - left;
                const long hi = (right < 0 || i + right > Lk - 1) ? Lk - 1 : i + right;
                double *p_row = P ? P + r * Lk : NULL;
                attend_row(Q + i * D, K + lo * D, V + lo * D, hi - lo + 1, D, hi - lo + 1, scale,
                           S, Pr, O + r * D, LSE + r, p_row ? p_row + lo : NULL);
                if (p_row)
                    for (long j = 0; j < lo; ++j) p_row[j] = 0.0;
                if (p_row)
                    for (long j = hi + 1; j < Lk; ++j) p_row[j] = 0.0;
            }
        }
        free(S);
        free(Pr);
    }
    return status;
}

/*
 * Key-padding mask on top of the band: query row i of a head whose batch has kv_len
 * valid keys may attend to key j iff  i - left <= j <= i + right  (as in
 * oracle_attn_head_window, -1 = unbounded) and  j < kv_len  (keys at or past kv_len
 * are padding).  This is one of the mask variants that the "FlashAttention-2 forward
 * in Triton" post (wsisp.com) leaves to later work.  A row whose allowed set is
 * empty -- kv_len = 0, or a band that lies entirely in the padding -- has no softmax;
 * the reading taken for it is O = 0 and LSE = -infinity (the log of an empty sum).
 * kv_len is clamped to [0, Lk].  Arguments otherwise as oracle_attn_head_window.
 */
int oracle_attn_head_keypad(const double *Q, const double *K, const double *V,
                            long Lq, long Lk, long D, long left, long right, long kv_len,
                            double scale, const long *rows, long nrows,
                            double *O, double *LSE, double *P, int nthreads)
{
    if (!Q || !K || !V || !O || !LSE) return ORACLE_BAD_ARG;
    if (Lq < 0 || Lk < 1 || D < 1 || nrows < 0 || left < -1 || right < -1) return ORACLE_BAD_ARG;
    if (!rows && nrows != Lq) return ORACLE_BAD_ARG;
    if (rows)
        for (long r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= Lq) return ORACLE_BAD_ARG;
    const long kv = kv_len < 0 ? 0 : (kv_len > Lk ? Lk : kv_len);
    int status = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)Lk);
        double *Pr = (double *)malloc(sizeof(double) * (size_t)Lk);
        const int have = S && Pr;
        if (!have) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_NO_MEMORY;
        }
        /* Every thread of the team meets the worksharing loop; one without its row
         * buffers takes its share of rows and skips them (the call then fails). */
        {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (long r = 0; r < nrows; ++r) {
                if (!have) continue;
                const long i = rows ? rows[r] : r;
                const long lo = (left < 0 || i - left < 0) ? 0 : i - left;
                long hi = (right < 0 || i + right > Lk - 1) ? Lk - 1 : i + right;
                if (hi > kv - 1) hi = kv - 1;
                double *p_row = P ? P + r * Lk : NULL;
                if (lo > hi) {   /* no allowed key: O = 0, LSE = -inf */
                    for (long d = 0; d < D; ++d) O[r * D + d] = 0.0;
                    LSE[r] = -INFINITY;
                    if (p_row)
                        for (long j = 0; j < Lk; ++j) p_row[j] = 0.0;
                    continue;
                }
                attend_row(Q + i * D, K + lo * D, V + lo * D, hi - lo + 1, D, hi - lo + 1, scale,
                           S, Pr, O + r * D, LSE + r, p_row ? p_row + lo : NULL);
                if (p_row) {
                    for (long j = 0; j < lo; ++j) p_row[j] = 0.0;
                    for (long j = hi + 1; j < Lk; ++j) p_row[j] = 0.0;
                }
            }
        }
        free(S);
        free(Pr);
    }
    return status;
}

/*
 * Gradients of the attention of one (batch, head) slice -- the backward pass that
 * the "FlashAttention-2 forward in Triton" post (wsisp.com) leaves to later work
 * and whose principle it states: recompute the probabilities rather than store
 * them.  With the loss's gradient dO with respect to O given, the chain rule
 * through O = P V, P = softmax_rows(S), S = scale Q K^T gives, per row i over its
 * allowed keys j (the same keys as oracle_attn_head):
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)      (the softmax Jacobian)
 *   dQ_i  = scale sum_j dS_ij K_j
 *   dK_j  = scale sum_i dS_ij Q_i
 * and 0 for every masked pair.  P and dS are materialised as [Lq, Lk] matrices
 * in double precision; dQ is formed per row, dV and dK per key row.
 *   Q, dO: [Lq, D]; K, V: [Lk, D]; dQ: [Lq, D]; dK, dV: [Lk, D] (all written).
 * Returns ORACLE_OK, ORACLE_BAD_ARG or ORACLE_NO_MEMORY.
 */
int oracle_attn_bwd_head(const double *Q, const double *K, const double *V, const double *dO,
                         long Lq, long Lk, long D, int causal, double scale,
                         double *dQ, double *dK, double *dV, int nthreads)
{
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV) return ORACLE_BAD_ARG;
    if (Lq < 0 || Lk < 1 || D < 1) return ORACLE_BAD_ARG;
    double *P = (double *)malloc(sizeof(double) * (size_t)(Lq > 0 ? Lq : 1) * (size_t)Lk);
    double *dS = (double *)malloc(sizeof(double) * (size_t)(Lq > 0 ? Lq : 1) * (size_t)Lk);
    if (!P || !dS) {
        free(P);
        free(dS);
        return ORACLE_NO_MEMORY;
    }
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (long i = 0; i < Lq; ++i) {
        const long n = allowed_keys(i, Lk, causal);
        double *p = P + i * Lk, *ds = dS + i * Lk;
        /* forward probabilities of row i, straight from the definition */
        double m = -INFINITY;
        for (long j = 0; j < n; ++j) {
            double dot = 0.0;
            for (long d = 0; d < D; ++d) dot += Q[i * D + d] * K[j * D + d];
            p[j] = scale * dot;
            if (p[j] > m) m = p[j];
        }
        double l = 0.0;
        for (long j = 0; j < n; ++j) {
            p[j] = exp(p[j] - m);
            l += p[j];
        }
        for (long j = 0; j < n; ++j) p[j] /= l;
        for (long j = n; j < Lk; ++j) p[j] = 0.0;
        /* dP_ij = dO_i . V_j, and the row's sum of P dP */
        double pdp = 0.0;
        for (long j = 0; j < n; ++j) {
            double dot = 0.0;
            for (long d = 0; d < D; ++d) dot += dO[i * D + d] * V[j * D + d];
            ds[j] = dot;
            pdp += p[j] * dot;
        }
        for (long j = 0; j < n; ++j) ds[j] = p[j] * (ds[j] - pdp);
        for (long j = n; j < Lk; ++j) ds[j] = 0.0;
        for (long d = 0; d < D; ++d) {
            double acc = 0.0;
            for (long j = 0; j < n; ++j) acc += ds[j] * K[j * D + d];
            dQ[i * D + d] = scale * acc;
        }
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (long j = 0; j < Lk; ++j) {
        for (long d = 0; d < D; ++d) {
            double av = 0.0, ak = 0.0;
            for (long i = 0; i < Lq; ++i) {
                av += P[i * Lk + j] * dO[i * D + d];
                ak += dS[i * Lk + j] * Q[i * D + d];
            }
            dV[j * D + d] = av;
            dK[j * D + d] = scale * ak;
        }
    }
    free(P);
    free(dS);
    return ORACLE_OK;
}

/* Allowed keys of query row i under the band (left, right; -1 = unbounded side) and the
 * key count kv: the contiguous range [*lo, *hi], empty when *lo > *hi. */
static void band_keys(long i, long Lk, long left, long right, long kv, long *lo, long *hi)
{
    *lo = (left < 0 || i - left < 0) ? 0 : i - left;
    long h = (right < 0 || i + right > Lk - 1) ? Lk - 1 : i + right;
    if (h > kv - 1) h = kv - 1;
    *hi = h;
}

/*
 * Gradients of one head at sampled outputs only, for heads too long for the Lq x Lk
 * matrices of oracle_attn_bwd_head(_masked): dQ at the query rows qrows[0..nq) and dK, dV
 * at the key rows krows[0..nk), by the same chain rule (P_ij = exp(scale Q_i.K_j - LSE_i),
 * dP_ij = dO_i.V_j, Delta_i = sum_j P_ij dP_ij, dS_ij = P_ij (dP_ij - Delta_i),
 * dQ_i = scale sum_j dS_ij K_j, dK_j = scale sum_i dS_ij Q_i, dV_j = sum_i P_ij dO_i) over
 * the allowed pairs of the band and key-padding mask of oracle_attn_bwd_head_masked (query
 * i sees keys i - left .. i + right below kv_len; -1 = unbounded side).  A row without
 * allowed keys has LSE = -inf, Delta = 0, dQ = 0 and adds nothing to dK, dV.  First every
 * query row's LSE_i and Delta_i are computed from the definition (O(Lq Lk D) work, one
 * score row of scratch per thread); then each sampled output is a sum over its row (dQ)
 * or its column (dK, dV).  LSE_all and Delta_all (Lq values each) receive the row
 * statistics when not NULL.
 */
int oracle_attn_bwd_rows_masked(const double *Q, const double *K, const double *V,
                                const double *dO, long Lq, long Lk, long D, long left,
                                long right, long kv_len, double scale, const long *qrows,
                                long nq, const long *krows, long nk, double *dQ_rows,
                                double *dK_rows, double *dV_rows, double *LSE_all,
                                double *Delta_all, int nthreads)
{
    if (!Q || !K || !V || !dO) return ORACLE_BAD_ARG;
    if (Lq < 1 || Lk < 1 || D < 1 || nq < 0 || nk < 0 || left < -1 || right < -1)
        return ORACLE_BAD_ARG;
    if ((nq > 0 && (!qrows || !dQ_rows)) || (nk > 0 && (!krows || !dK_rows || !dV_rows)))
        return ORACLE_BAD_ARG;
    for (long r = 0; r < nq; ++r)
        if (qrows[r] < 0 || qrows[r] >= Lq) return ORACLE_BAD_ARG;
    for (long r = 0; r < nk; ++r)
        if (krows[r] < 0 || krows[r] >= Lk) return ORACLE_BAD_ARG;
    const long kv = kv_len < 0 ? 0 : (kv_len > Lk ? Lk : kv_len);
    double *lse = (double *)malloc(sizeof(double) * (size_t)Lq);
    double *delta = (double *)malloc(sizeof(double) * (size_t)Lq);
    if (!lse || !delta) {
        free(lse);
        free(delta);
        return ORACLE_NO_MEMORY;
    }
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *srow = (double *)malloc(sizeof(double) * (size_t)Lk);
        if (!srow) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 8)
#endif
        for (long i = 0; i < Lq; ++i) {
            if (!srow) continue;
            long lo, hi;
            band_keys(i, Lk, left, right, kv, &lo, &hi);
            if (lo > hi) {   /* no allowed key */
                lse[i] = -INFINITY;
                delta[i] = 0.0;
                continue;
            }
            double m = -INFINITY;
            for (long j = lo; j <= hi; ++j) {
                double dot = 0.0;
                for (long d = 0; d < D; ++d) dot += Q[i * D + d] * K[j * D + d];
                srow[j] = scale * dot;
                if (srow[j] > m) m = srow[j];
            }
            double l = 0.0;
            for (long j = lo; j <= hi; ++j) l += exp(srow[j] - m);
            const double lse_i = m + log(l);
            double pdp = 0.0;
            for (long j = lo; j <= hi; ++j) {
                double dot = 0.0;
                for (long d = 0; d < D; ++d) dot += dO[i * D + d] * V[j * D + d];
                pdp += exp(srow[j] - lse_i) * dot;
            }
            lse[i] = lse_i;
            delta[i] = pdp;
        }
        free(srow);
    }
    if (bad) {
        free(lse);
        free(delta);
        return ORACLE_NO_MEMORY;
    }
    /* dQ at the sampled query rows: sums over the row's allowed keys */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long r = 0; r < nq; ++r) {
        const long i = qrows[r];
        long lo, hi;
        band_keys(i, Lk, left, right, kv, &lo, &hi);
        double *out = dQ_rows + r * D;
        for (long d = 0; d < D; ++d) out[d] = 0.0;
        for (long j = lo; j <= hi; ++j) {
            double s = 0.0, dp = 0.0;
            for (long d = 0; d < D; ++d) {
                s += Q[i * D + d] * K[j * D + d];
                dp += dO[i * D + d] * V[j * D + d];
            }
            const double p = exp(scale * s - lse[i]);
            const double ds = p * (dp - delta[i]);
            for (long d = 0; d < D; ++d) out[d] += ds * K[j * D + d];
        }
        for (long d = 0; d < D; ++d) out[d] *= scale;
    }
    /* dK, dV at the sampled key rows: sums over the queries that see the key */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long r = 0; r < nk; ++r) {
        const long j = krows[r];
        double *ok = dK_rows + r * D, *ov = dV_rows + r * D;
        for (long d = 0; d < D; ++d) ok[d] = ov[d] = 0.0;
        for (long i = 0; i < Lq; ++i) {
            long lo, hi;
            band_keys(i, Lk, left, right, kv, &lo, &hi);
            if (j < lo || j > hi) continue;
            double s = 0.0, dp = 0.0;
            for (long d = 0; d < D; ++d) {
                s += Q[i * D + d] * K[j * D + d];
                dp += dO[i * D + d] * V[j * D + d];
            }
            const double p = exp(scale * s - lse[i]);
            const double ds = p * (dp - delta[i]);
            for (long d = 0; d < D; ++d) {
                ov[d] += p * dO[i * D + d];
                ok[d] += ds * Q[i * D + d];
            }
        }
        for (long d = 0; d < D; ++d) ok[d] *= scale;
    }
    if (LSE_all)
        for (long i = 0; i < Lq; ++i) LSE_all[i] = lse[i];
    if (Delta_all)
        for (long i = 0; i < Lq; ++i) Delta_all[i] = delta[i];
    free(lse);
    free(delta);
    return ORACLE_OK;
}

/* oracle_attn_bwd_rows_masked for the causal mask (band (-1, 0): key j <= i) or the full
 * mask (band (-1, -1)), no key padding. */
int oracle_attn_bwd_rows(const double *Q, const double *K, const double *V, const double *dO,
                         long Lq, long Lk, long D, int causal, double scale,
                         const long *qrows, long nq, const long *krows, long nk,
                         double *dQ_rows, double *dK_rows, double *dV_rows,
                         double *LSE_all, double *Delta_all, int nthreads)
{
    return oracle_attn_bwd_rows_masked(Q, K, V, dO, Lq, Lk, D, -1, causal ? 0 : -1, Lk, scale,
                                       qrows, nq, krows, nk, dQ_rows, dK_rows, dV_rows, LSE_all,
                                       Delta_all, nthreads);
}

/*
 * Gradients under the band and key-padding mask of oracle_attn_head_keypad: the same
 * chain rule as oracle_attn_bwd_head, with row i's allowed keys the contiguous range
 * [lo_i, hi_i] (i - left <= j <= i + right, j < kv_len; -1 = unbounded side) instead of
 * a prefix.  A row without allowed keys has O = 0 (not a function of Q, K or V), so it
 * contributes nothing: dQ_i = 0 and no term to dK or dV.  kv_len is clamped to [0, Lk].
 */
int oracle_attn_bwd_head_masked(const double *Q, const double *K, const double *V,
                                const double *dO, long Lq, long Lk, long D, long left,
                                long right, long kv_len, double scale, double *dQ, double *dK,
                                double *dV, int nthreads)
{
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV) return ORACLE_BAD_ARG;
    if (Lq < 0 || Lk < 1 || D < 1 || left < -1 || right < -1) return ORACLE_BAD_ARG;
    const long kv = kv_len < 0 ? 0 : (kv_len > Lk ? Lk : kv_len);
    double *P = (double *)calloc((size_t)(Lq > 0 ? Lq : 1) * (size_t)Lk, sizeof(double));
    double *dS = (double *)calloc((size_t)(Lq > 0 ? Lq : 1) * (size_t)Lk, sizeof(double));
    if (!P || !dS) {
        free(P);
        free(dS);
        return ORACLE_NO_MEMORY;
    }
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads)
#endif
    for (long i = 0; i < Lq; ++i) {
        const long lo = (left < 0 || i - left < 0) ? 0 : i - left;
        long hi = (right < 0 || i + right > Lk - 1) ? Lk - 1 : i + right;
        if (hi > kv - 1) hi = kv - 1;
        double *p = P + i * Lk, *ds = dS + i * Lk;
        for (long d = 0; d < D; ++d) dQ[i * D + d] = 0.0;
        if (lo > hi) continue;   /* no allowed key: P and dS stay 0 */
        double m = -INFINITY;
        for (long j = lo; j <= hi; ++j) {
            double dot = 0.0;
            for (long d = 0; d < D; ++d) dot += Q[i * D + d] * K[j * D + d];
            p[j] = scale * dot;
            if (p[j] > m) m = p[j];
        }
        double l = 0.0;
        for (long j = lo; j <= hi; ++j) {
            p[j] = exp(p[j] - m);
            l += p[j];
        }
        for (long j = lo; j <= hi; ++j) p[j] /= l;
        double pdp = 0.0;
        for (long j = lo; j <= hi; ++j) {
            double dot = 0.0;
            for (long d = 0; d < D; ++d) dot += dO[i * D + d] * V[j * D + d];
            ds[j] = dot;
            pdp += p[j] * dot;
        }
        for (long j = lo; j <= hi; ++j) ds[j] = p[j] * (ds[j] - pdp);
        for (long d = 0; d < D; ++d) {
            double acc = 0.0;
            for (long j = lo; j <= hi; ++j) acc += ds[j] * K[j * D + d];
            dQ[i * D + d] = scale * acc;
        }
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (long j = 0; j < Lk; ++j) {
        for (long d = 0; d < D; ++d) {
            double av = 0.0, ak = 0.0;
            for (long i = 0; i < Lq; ++i) {
                av += P[i * Lk + j] * dO[i * D + d];
                ak += dS[i * Lk + j] * Q[i * D + d];
            }
            dV[j * D + d] = av;
            dK[j * D + d] = scale * ak;
        }
    }
    free(P);
    free(dS);
    return ORACLE_OK;
}

/* Threads the OpenMP runtime would use by default (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
