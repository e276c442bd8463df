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
 * Returns ORACLE_OK, or an error code with no output written.
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
        if (!S || !Pr) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_NO_MEMORY;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (long r = 0; r < nrows; ++r) {
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
        if (!S || !Pr) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_NO_MEMORY;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
            for (long r = 0; r < nrows; ++r) {
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

/* Threads the OpenMP runtime would use by default (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
