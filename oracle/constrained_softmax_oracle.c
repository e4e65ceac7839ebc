/*
 * Oracle for the entropy-bounded softmax ("constrained_softmax").
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously correct
 * CPU statement of what the method computes.  Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark load it.  The CUDA library
 * shares no code, header, table or helper with it, and neither side calls the
 * other.
 *
 * Source of the method: "BURT-IMMA CUDA Kernel API Reference", section 2.1
 * `constrained_softmax` (Parameters table, Description steps 1-4, Performance
 * Notes) and section 5 (5.1 Error Codes, 5.3 NaN/Inf Propagation Policy,
 * 5.4 Graceful Degradation); the backward follows section 6.3 (PyTorch Custom
 * Op Integration, ConstrainedSoftmaxFunction.backward) with the 1/T of
 * softmax(l / T) restored; attention_softmax follows section 2.6 and
 * biencoder_attention section 2.5.
 *
 * Arithmetic: IEEE double throughout, libm exp() and log().  The fp32
 * parameters are promoted exactly to double, so both sides of any comparison
 * see the same bound (0.2f is 0.20000000298... here as on the GPU).
 *
 * Readings of the page where it is silent or loose (all stated again in the
 * design notes):
 *  - Description step 1 divides by T before any T exists: the first softmax
 *    is the standard one, T = 1.
 *  - The search (step 3) runs only when H(1) > entropy_bound.  Entropy is
 *    nondecreasing in T (step 4 says lower T concentrates the distribution),
 *    so temperatures above 1 can never help; the search interval is
 *    [temperature_min, min(1, temperature_max)].
 *  - Step 3 aims at "H = entropy_bound" while the section heading asks for
 *    H(p) <= entropy_bound: the search keeps the feasible end `lo` (ties go
 *    to lo) and the output is softmax(l / lo).
 *  - "Number of binary search iterations": exactly max_iterations halvings,
 *    no early exit.  When temperature_min >= min(1, temperature_max) there is
 *    no interval to halve and T = temperature_min.
 *  - 5.3: a NaN or an Inf anywhere in a row affects every p_i of that row, so
 *    the whole row is zeroed, T is reported as NaN and the row's flag is
 *    NAN_INPUT (1) or INF_INPUT (2); NaN wins when both occur.
 *  - 5.4: an unsatisfiable bound returns the lowest achievable entropy, which
 *    is softmax at T = temperature_min, with flag ENTROPY_OVERFLOW (3).
 */
#include <math.h>
#include <stdint.h>

/* Flag values: section 5.1, enum BurtError. */
#define ORACLE_FLAG_NONE 0
#define ORACLE_FLAG_NAN_INPUT 1
#define ORACLE_FLAG_INF_INPUT 2
#define ORACLE_FLAG_ENTROPY_OVERFLOW 3

/* Largest logit of the row (the max-subtraction that keeps exp() finite;
 * softmax is unchanged by subtracting a constant from every logit). */
static double row_max(const float* l, int64_t C)
{
    double m = (double)l[0];
    for (int64_t i = 1; i < C; ++i) {
        if ((double)l[i] > m) m = (double)l[i];
    }
    return m;
}

/* p = softmax(l / T): Description step 1, p_i = exp(l_i/T) / sum_j exp(l_j/T). */
static void softmax_at(const float* l, int64_t C, double T, double* p)
{
    double m = row_max(l, C);
    double S = 0.0;
    for (int64_t i = 0; i < C; ++i) {
        S += exp(((double)l[i] - m) / T);
    }
    for (int64_t i = 0; i < C; ++i) {
        p[i] = exp(((double)l[i] - m) / T) / S;
    }
}

/* H(T) = -sum_i p_i ln p_i with p = softmax(l / T), in nats (Description
 * step 2; the Parameters table gives the bound in nats).  A term with
 * p_i = 0 contributes 0 (the limit of p ln p). */
static double entropy_at(const float* l, int64_t C, double T)
{
    double m = row_max(l, C);
    double S = 0.0;
    for (int64_t i = 0; i < C; ++i) {
        S += exp(((double)l[i] - m) / T);
    }
    double H = 0.0;
    for (int64_t i = 0; i < C; ++i) {
        double p = exp(((double)l[i] - m) / T) / S;
        if (p > 0.0) H -= p * log(p);
    }
    return H;
}

/* Public: H(T) of one row, for pinning the oracle against closed forms. */
double oracle_entropy(const float* l, int64_t C, double T)
{
    return entropy_at(l, C, T);
}

/* Public: softmax(l / T) of one row. */
void oracle_softmax(const float* l, int64_t C, double T, double* p)
{
    softmax_at(l, C, T, p);
}

/*
 * One row of constrained_softmax.  Writes C probabilities to p and returns
 * the flag; *T_out gets the temperature used, *iters_out the number of
 * bisection steps taken (each step evaluates H once).  If path_mid/path_H are
 * non-NULL they receive the midpoint and H(midpoint) of every step.
 */
static int one_row(const float* l, int64_t C, double bound, double t_min,
                   double t_max, int32_t max_iter, double* p, double* T_out,
                   int32_t* iters_out, double* path_mid, double* path_H)
{
    int has_nan = 0, has_inf = 0;
    for (int64_t i = 0; i < C; ++i) {
        if (isnan(l[i])) has_nan = 1;
        else if (isinf(l[i])) has_inf = 1;
    }
    *iters_out = 0;
    if (has_nan || has_inf) {
        for (int64_t i = 0; i < C; ++i) p[i] = 0.0;
        *T_out = NAN;
        return has_nan ? ORACLE_FLAG_NAN_INPUT : ORACLE_FLAG_INF_INPUT;
    }

    /* Steps 1-2: standard softmax and its entropy. */
    if (entropy_at(l, C, 1.0) <= bound) {
        softmax_at(l, C, 1.0, p);
        *T_out = 1.0;
        return ORACLE_FLAG_NONE;
    }

    /* Step 3: bisection on T over [t_min, min(1, t_max)]. */
    double lo = t_min;
    double hi = t_max < 1.0 ? t_max : 1.0;
    if (lo < hi) {
        for (int32_t k = 0; k < max_iter; ++k) {
            double mid = (lo + hi) / 2.0;
            double Hmid = entropy_at(l, C, mid);
            if (path_mid) path_mid[k] = mid;
            if (path_H) path_H[k] = Hmid;
            if (Hmid > bound) {
                hi = mid;
            } else {
                lo = mid;
            }
        }
        *iters_out = max_iter;
    }

    softmax_at(l, C, lo, p);
    *T_out = lo;
    /* 5.4: only lo = t_min can still violate the bound. */
    if (entropy_at(l, C, lo) > bound) return ORACLE_FLAG_ENTROPY_OVERFLOW;
    return ORACLE_FLAG_NONE;
}

/*
 * Rows [row_begin, row_end) of a row-major [batch, C] fp32 logit matrix.
 * out is [batch, C] double; T_out, flags_out and iters_out are [batch].
 * Rows are independent, so callers may split a batch over threads.
 */
void oracle_constrained_softmax_rows(const float* logits, double* out,
                                     int64_t row_begin, int64_t row_end,
                                     int64_t C, float entropy_bound,
                                     float t_min, float t_max,
                                     int32_t max_iter, double* T_out,
                                     int32_t* flags_out, int32_t* iters_out)
{
    for (int64_t b = row_begin; b < row_end; ++b) {
        flags_out[b] = one_row(logits + b * C, C, (double)entropy_bound,
                               (double)t_min, (double)t_max, max_iter,
                               out + b * C, &T_out[b], &iters_out[b], 0, 0);
    }
}

/* One row with its bisection path recorded (max_iter entries each). */
int32_t oracle_constrained_softmax_path(const float* l, double* p, int64_t C,
                                        float entropy_bound, float t_min,
                                        float t_max, int32_t max_iter,
                                        double* T_out, int32_t* iters_out,
                                        double* path_mid, double* path_H)
{
    return one_row(l, C, (double)entropy_bound, (double)t_min, (double)t_max,
                   max_iter, p, T_out, iters_out, path_mid, path_H);
}

/*
 * Backward of constrained_softmax: the vector-Jacobian product of section
 * 6.3 (ConstrainedSoftmaxFunction.backward) with the temperature restored.
 *
 * The output is p = softmax(l / T), where T is the bisection's final lo.
 * That lo is one of finitely many grid points chosen by the comparisons
 * H(mid) > bound, so T is piecewise constant in l: its derivative is zero
 * everywhere except on the measure-zero set where a comparison flips.  There
 * dp_i/dl_k = (1/T) p_i (delta_ik - p_k), and for an upstream gradient g
 *
 *     grad_k = sum_i g_i dp_i/dl_k = (1/T) p_k (g_k - sum_i g_i p_i).
 *
 * Section 6.3 writes p (g - <g, p>): the same product without the 1/T, which
 * is exact only where T = 1.  A row whose T is not a positive finite number
 * (NaN: section 5.3 zeroed the row, so its output does not depend on l) gets
 * a zero gradient.
 *
 * p, g and grad are row-major [*, C] doubles, T is [*]; rows
 * [row_begin, row_end) are computed.
 */
void oracle_constrained_softmax_backward_rows(const double* p, const double* g,
                                              const double* T, double* grad,
                                              int64_t row_begin,
                                              int64_t row_end, int64_t C)
{
    for (int64_t b = row_begin; b < row_end; ++b) {
        const double* pb = p + b * C;
        const double* gb = g + b * C;
        double* out = grad + b * C;
        if (!(T[b] > 0.0) || isinf(T[b])) {
            for (int64_t k = 0; k < C; ++k) out[k] = 0.0;
            continue;
        }
        double dot = 0.0;
        for (int64_t i = 0; i < C; ++i) dot += gb[i] * pb[i];
        for (int64_t k = 0; k < C; ++k) out[k] = pb[k] * (gb[k] - dot) / T[b];
    }
}

/*
 * attention_softmax: section 2.6 (Signature, Parameters table, Description
 * steps 1-3).  scores is row-major [B, H, S, S]; row r = ((b H) + h) S + i
 * holds the scores of query i against keys j = 0..S-1.  mask is NULL or
 * [B, S] (the page's [B, 1, 1, S]), added to every row of batch b.
 *
 *  1. v_j = scores[r, j] + mask[b, j], added in fp32 (the inputs' precision,
 *     as the page's fp32 kernel adds them); a mask of -inf removes key j;
 *  2. causal: keys j > i are removed (their scores are never used);
 *  3. p = softmax over the kept keys with the max subtracted (fp64 here),
 *     p_j = 0 for removed keys.
 *
 * Readings (stated again in the design notes):
 *  - section 5.3 applies to the scores and the mask the row uses: a NaN
 *    (flag 1) or an infinity (flag 2; a mask of -inf is the masking value,
 *    not an error) zeroes the whole row; NaN wins over Inf;
 *  - a row whose keys are all removed has no distribution: zeros, flag 0.
 */
/* Step 1: the score plus the mask, added in fp32. */
static double masked_score(const float* s, const float* m, int64_t j)
{
    if (!m) return (double)s[j];
    const float v = s[j] + m[j];
    return (double)v;
}

/* One row: query i against keys 0..S-1; s the row's scores, m the batch's
 * mask row or NULL; writes p[0..S) and returns the flag. */
static int32_t attention_row(const float* s, const float* m, int64_t S,
                             int64_t i, int32_t causal, double* p)
{
    /* Step 2: keys j > i are removed from a causal row. */
    const int64_t kept_end = causal ? i + 1 : S;
    int has_nan = 0, has_inf = 0;
    for (int64_t j = 0; j < kept_end; ++j) {
        if (isnan(s[j])) has_nan = 1;
        else if (isinf(s[j])) has_inf = 1;
        if (m) {
            if (isnan(m[j])) has_nan = 1;
            else if (isinf(m[j]) && m[j] > 0) has_inf = 1;
        }
    }
    for (int64_t j = 0; j < S; ++j) p[j] = 0.0;
    if (has_nan || has_inf)
        return has_nan ? ORACLE_FLAG_NAN_INPUT : ORACLE_FLAG_INF_INPUT;
    /* Step 3: softmax over the kept keys (a -inf value is a removed key
     * and contributes exp(-inf) = 0). */
    double vmax = -INFINITY;
    for (int64_t j = 0; j < kept_end; ++j) {
        const double v = masked_score(s, m, j);
        if (v > vmax) vmax = v;
    }
    if (vmax == -INFINITY) return ORACLE_FLAG_NONE;   /* every key removed */
    double sum = 0.0;
    for (int64_t j = 0; j < kept_end; ++j) {
        p[j] = exp(masked_score(s, m, j) - vmax);
        sum += p[j];
    }
    for (int64_t j = 0; j < kept_end; ++j) p[j] /= sum;
    return ORACLE_FLAG_NONE;
}

void oracle_attention_softmax_rows(const float* scores, const float* mask,
                                   double* out, int64_t row_begin,
                                   int64_t row_end, int64_t H, int64_t S,
                                   int32_t causal, int32_t* flags_out)
{
    for (int64_t r = row_begin; r < row_end; ++r) {
        const int64_t b = r / (H * S);
        const int64_t i = r % S;
        const float* m = mask ? mask + b * S : 0;
        flags_out[r] = attention_row(scores + r * S, m, S, i, causal,
                                     out + r * S);
    }
}

/* Public: one row given its query index i (for sampled rows of launches
 * too large to recompute whole). */
int32_t oracle_attention_softmax_row(const float* s, const float* m,
                                     int64_t S, int64_t i, int32_t causal,
                                     double* p)
{
    return attention_row(s, m, S, i, causal, p);
}

/*
 * biencoder_attention: section 2.5 (Signature, Parameters table,
 * Description steps 1-3).  query [BH, Q, D], keys and values [BH, K, D]
 * (BH = batch x heads), all row-major fp32.
 *
 * Step 1, scores = query @ keys^T * scale.  The page's kernel is fp32 and
 * the constrained softmax's search turns its logits into a grid index, so
 * the scores are fixed to one fp32 evaluation (the reading stated in the
 * design notes): s = sum over d = 0..D-1 of q_d k_d, accumulated with one
 * fused multiply-add per term in that order from 0, then one fp32 multiply
 * by scale.  Steps 2-3 (the constrained softmax of each row of scores and
 * attn @ values) are computed in fp64 by the caller from these scores.
 */
void oracle_biencoder_scores(const float* q, const float* k, float* scores,
                             int64_t BH, int64_t Q, int64_t K, int64_t D,
                             float scale)
{
    for (int64_t bh = 0; bh < BH; ++bh) {
        for (int64_t i = 0; i < Q; ++i) {
            const float* qi = q + (bh * Q + i) * D;
            for (int64_t j = 0; j < K; ++j) {
                const float* kj = k + (bh * K + j) * D;
                float s = 0.0f;
                for (int64_t d = 0; d < D; ++d) s = fmaf(qi[d], kj[d], s);
                scores[(bh * Q + i) * K + j] = s * scale;
            }
        }
    }
}
