/*
 * sdpa_oracle.c -- plain, slow, fp64 CPU oracle for the materialised-probability
 * scaled-dot-product-attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the tests, the smoke check and the CPU-baseline leg of the benchmark do.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes (FlagOS-OP PR #10 "feat: add sdpa_math operator",
 * overview and "semantics" items):
 *   the math backend of SDPA returns both the output and the full probability
 *   map, (O, P), with
 *       s[i,j] = scale * sum_d q[b,h,i,d] * k[b,hk,j,d]        (hk = h / (Hq/Hkv))
 *       s[i,j] = -inf  if is_causal and j > i                  (top-left causal)
 *       s[i,j] = -inf  if a bool mask holds false at [i,j]     (-inf masking, as F.sdpa)
 *       s[i,j] += m[i,j] for an additive (float) mask
 *       P[i,:] = softmax_j(s[i,:]),   O[i,:] = sum_j P[i,j] * v[b,hk,j,:]
 *   and fixes four semantics:
 *     - is_causal together with an attn_mask is an error;
 *     - a row with every key masked gives P = 0 and O = 0 (not NaN);
 *     - Hq not divisible by Hkv is an error (GQA);
 *     - dropout is not part of this path (dropout_p = 0).
 *
 * The softmax is evaluated by its textbook definition: subtract the row max,
 * exponentiate, divide by the sum.  Everything is double precision; inputs are
 * the exact values of the caller's dtype widened to double.  The log-sum-exp of
 * each row (max + log(sum)) is returned for diagnostics; -inf for a fully
 * masked row.
 *
 * Pins: every function here is checked by CPU tests against closed forms,
 * invariants, brute force on tiny inputs and an independent float64 library
 * evaluation (softmax + matmul; for the backward, central finite differences
 * of the forward and float64 autograd).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARGUMENT 1

#define MASK_NONE 0
#define MASK_BOOL 1
#define MASK_ADDITIVE 2

/* One query row: (b, h, i).  Writes Dv outputs, Skv probabilities and the lse.
 * `s` is caller-provided scratch of Skv doubles. */
static void oracle_one_row(const double *q, const double *k, const double *v,
                           const double *mask, int mask_kind, int64_t mask_b,
                           int64_t mask_h, int64_t Hq, int64_t Hkv, int64_t Sq,
                           int64_t Skv, int64_t D, int64_t Dv, int is_causal,
                           double scale, int64_t b, int64_t h, int64_t i,
                           double *o_row, double *p_row, double *lse_out,
                           double *s) {
    const int64_t group = Hq / Hkv;
    const int64_t hk = h / group; /* query head h reads key/value head h / group */
    const double *qi = q + ((b * Hq + h) * Sq + i) * D;
    const double *kb = k + (b * Hkv + hk) * Skv * D;
    const double *vb = v + (b * Hkv + hk) * Skv * Dv;
    const double *mrow = NULL;
    if (mask_kind != MASK_NONE) {
        /* the mask broadcasts over batch and head when its extent there is 1 */
        const int64_t mb = (mask_b == 1) ? 0 : b;
        const int64_t mh = (mask_h == 1) ? 0 : h;
        mrow = mask + ((mb * mask_h + mh) * Sq + i) * Skv;
    }

    /* scores, with causal / bool / additive masking */
    for (int64_t j = 0; j < Skv; ++j) {
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) acc += qi[d] * kb[j * D + d];
        double sj = scale * acc;
        if (is_causal && j > i) sj = -INFINITY;
        if (mask_kind == MASK_BOOL && mrow[j] == 0.0) sj = -INFINITY;
        if (mask_kind == MASK_ADDITIVE) sj += mrow[j];
        s[j] = sj;
    }

    /* row max; a row whose max is -inf (or with no keys at all) is fully masked */
    double m = -INFINITY;
    for (int64_t j = 0; j < Skv; ++j)
        if (s[j] > m) m = s[j];

    if (Skv == 0 || m == -INFINITY) {
        for (int64_t j = 0; j < Skv; ++j) p_row[j] = 0.0;
        for (int64_t e = 0; e < Dv; ++e) o_row[e] = 0.0;
        *lse_out = -INFINITY;
        return;
    }

    /* softmax by definition: exp(s - max) / sum */
    double z = 0.0;
    for (int64_t j = 0; j < Skv; ++j) {
        double ej = exp(s[j] - m); /* exp(-inf) == 0 for masked keys */
        p_row[j] = ej;
        z += ej;
    }
    for (int64_t j = 0; j < Skv; ++j) p_row[j] /= z;
    *lse_out = m + log(z);

    /* O = P V */
    for (int64_t e = 0; e < Dv; ++e) o_row[e] = 0.0;
    for (int64_t j = 0; j < Skv; ++j) {
        const double pj = p_row[j];
        if (pj == 0.0) continue; /* a masked key contributes nothing */
        for (int64_t e = 0; e < Dv; ++e) o_row[e] += pj * vb[j * Dv + e];
    }
}

/*
 * sdpa_oracle_fwd -- the oracle entry point.
 *
 *   q    [B, Hq,  Sq,  D ]  contiguous doubles
 *   k    [B, Hkv, Skv, D ]  contiguous doubles
 *   v    [B, Hkv, Skv, Dv]  contiguous doubles
 *   mask [mask_b, mask_h, Sq, Skv] contiguous doubles, or NULL when mask_kind
 *        is MASK_NONE.  mask_b is 1 or B, mask_h is 1 or Hq (broadcast).
 *        For MASK_BOOL a value of 0 masks the key (-inf), any other keeps it.
 *   rows  optional list of flattened row ids ((b*Hq + h)*Sq + i); when NULL
 *         every row is computed in order and nrows must be B*Hq*Sq.
 *   out   [nrows, Dv], probs [nrows, Skv], lse [nrows]   (outputs, doubles)
 *   nthreads  OpenMP threads (1 = serial).  Rows are independent, so the
 *             result does not depend on the thread count.
 *
 * Returns ORACLE_OK, or ORACLE_ERR_ARGUMENT for: Hq % Hkv != 0, causal with a
 * mask, a bad mask broadcast extent, a negative size or an out-of-range row id.
 */
int sdpa_oracle_fwd(const double *q, const double *k, const double *v,
                    const double *mask, int mask_kind, int64_t mask_b,
                    int64_t mask_h, int64_t B, int64_t Hq, int64_t Hkv,
                    int64_t Sq, int64_t Skv, int64_t D, int64_t Dv,
                    int is_causal, double scale, const int64_t *rows,
                    int64_t nrows, double *out, double *probs, double *lse,
                    int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv < 0 || D < 0 || Dv < 0)
        return ORACLE_ERR_ARGUMENT;
    if (Hq % Hkv != 0) return ORACLE_ERR_ARGUMENT;          /* GQA divisibility */
    if (is_causal && mask_kind != MASK_NONE) return ORACLE_ERR_ARGUMENT;
    if (mask_kind != MASK_NONE && mask_kind != MASK_BOOL && mask_kind != MASK_ADDITIVE)
        return ORACLE_ERR_ARGUMENT;
    if (mask_kind != MASK_NONE) {
        if (mask == NULL) return ORACLE_ERR_ARGUMENT;
        if (!(mask_b == 1 || mask_b == B) || !(mask_h == 1 || mask_h == Hq))
            return ORACLE_ERR_ARGUMENT;
    }
    const int64_t total = B * Hq * Sq;
    if (rows == NULL && nrows != total) return ORACLE_ERR_ARGUMENT;
    if (rows != NULL)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= total) return ORACLE_ERR_ARGUMENT;
    if (nthreads < 1) nthreads = 1;

    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *s = (double *)malloc((size_t)(Skv > 0 ? Skv : 1) * sizeof(double));
        if (s == NULL) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
        for (int64_t r = 0; r < nrows; ++r) {
            if (s == NULL) continue;
            const int64_t id = rows ? rows[r] : r;
            const int64_t i = id % Sq;
            const int64_t h = (id / Sq) % Hq;
            const int64_t b = id / (Sq * Hq);
            oracle_one_row(q, k, v, mask, mask_kind, mask_b, mask_h, Hq, Hkv, Sq,
                           Skv, D, Dv, is_causal, scale, b, h, i, out + r * Dv,
                           probs + r * Skv, lse + r, s);
        }
        free(s);
    }
    return failed ? ORACLE_ERR_ARGUMENT : ORACLE_OK;
}

/*
 * sdpa_oracle_bwd -- gradients of the (O, P) forward, given its probability map.
 *
 * What it computes (FlagOS-OP PR #10: the overview's A1 item, where gradients
 * flow through both outputs, dout and dprobs; the "2026-10-07 update: P800
 * fused backward", where dprobs goes through the exact softmax Jacobian of the
 * materialised probability map and GQA query / key gradients are reduced back
 * to the KV heads).  For the scalar L = sum(O * dout) + sum(P * dprobs) with
 * (O, P) the forward of (q, k, v), per (b, h, i), hk = h / (Hq / Hkv):
 *     dP[i,j]  = sum_e dout[b,h,i,e] * v[b,hk,j,e] + dprobs[b,h,i,j]
 *     rsum[i]  = sum_j P[i,j] * dP[i,j]
 *     dS[i,j]  = P[i,j] * (dP[i,j] - rsum[i])        (softmax Jacobian)
 *     dq[b,h,i,:]   = scale * sum_j dS[i,j] * k[b,hk,j,:]
 *     dk[b,hk,j,:] += scale * dS[i,j] * q[b,h,i,:]    (summed over the group's heads)
 *     dv[b,hk,j,:] += P[i,j] * dout[b,h,i,:]          (summed over the group's heads)
 * Masked keys and fully masked rows have P = 0 and so no gradient; the mask
 * itself gets none.  All double precision; P is taken as given (the forward's).
 *
 *   q [B,Hq,Sq,D], k [B,Hkv,Skv,D], v [B,Hkv,Skv,Dv], probs [B,Hq,Sq,Skv],
 *   dout [B,Hq,Sq,Dv], dprobs [B,Hq,Sq,Skv] or NULL (no gradient through P);
 *   outputs dq [B,Hq,Sq,D], dk [B,Hkv,Skv,D], dv [B,Hkv,Skv,Dv] (overwritten).
 * Work is split over (b, hk): each owns its dk / dv rows, so the result does
 * not depend on the thread count.
 */
int sdpa_oracle_bwd(const double *q, const double *k, const double *v,
                    const double *probs, const double *dout, const double *dprobs,
                    int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Skv,
                    int64_t D, int64_t Dv, double scale, double *dq, double *dk,
                    double *dv, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Skv < 0 || D < 0 || Dv < 0)
        return ORACLE_ERR_ARGUMENT;
    if (Hq % Hkv != 0) return ORACLE_ERR_ARGUMENT;
    const int64_t g = Hq / Hkv;
    if (nthreads < 1) nthreads = 1;
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *dp = (double *)malloc((size_t)(Skv > 0 ? Skv : 1) * sizeof(double));
        if (dp == NULL) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t bk = 0; bk < B * Hkv; ++bk) {
            if (dp == NULL) continue;
            const int64_t b = bk / Hkv, hk = bk % Hkv;
            const double *kb = k + (b * Hkv + hk) * Skv * D;
            const double *vb = v + (b * Hkv + hk) * Skv * Dv;
            double *dkb = dk + (b * Hkv + hk) * Skv * D;
            double *dvb = dv + (b * Hkv + hk) * Skv * Dv;
            for (int64_t x = 0; x < Skv * D; ++x) dkb[x] = 0.0;
            for (int64_t x = 0; x < Skv * Dv; ++x) dvb[x] = 0.0;
            for (int64_t h = hk * g; h < (hk + 1) * g; ++h) {
                for (int64_t i = 0; i < Sq; ++i) {
                    const int64_t row = (b * Hq + h) * Sq + i;
                    const double *pr = probs + row * Skv;
                    const double *go = dout + row * Dv;
                    const double *qr = q + row * D;
                    double rsum = 0.0;
                    for (int64_t j = 0; j < Skv; ++j) {
                        double acc = dprobs ? dprobs[row * Skv + j] : 0.0;
                        for (int64_t e = 0; e < Dv; ++e) acc += go[e] * vb[j * Dv + e];
                        dp[j] = acc;
                        rsum += pr[j] * acc;
                    }
                    double *dqr = dq + row * D;
                    for (int64_t d = 0; d < D; ++d) dqr[d] = 0.0;
                    for (int64_t j = 0; j < Skv; ++j) {
                        const double ds = pr[j] * (dp[j] - rsum);
                        for (int64_t d = 0; d < D; ++d) {
                            dqr[d] += scale * ds * kb[j * D + d];
                            dkb[j * D + d] += scale * ds * qr[d];
                        }
                        for (int64_t e = 0; e < Dv; ++e) dvb[j * Dv + e] += pr[j] * go[e];
                    }
                }
            }
        }
        free(dp);
    }
    return failed ? ORACLE_ERR_ARGUMENT : ORACLE_OK;
}

/* Number of OpenMP threads the oracle would use by default (1 without OpenMP). */
int sdpa_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
