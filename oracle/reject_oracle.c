/*
 * reject_oracle.c -- plain fp64 CPU oracle of the verify-side rejection sampler.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; the two meet only in the seeded synthetic inputs.
 *
 * What it computes, step by step, in the order the pages give it:
 *
 *  - Per request r with k = cu[r+1]-cu[r] drafts, its k+1 target rows are
 *    t = cu[r]+r+i (i = 0..k) and its draft rows d = cu[r]+i (i < k): the ragged
 *    flattened layout of "第12章 投机解码：以小博大" §12.3.5 (draft_token_ids,
 *    num_draft_tokens, cu_num_draft_tokens, target and bonus logits indices) and
 *    "vllm v1 源码精读（五）" §8 (SpecDecodeMetadata).  k is capped at 32
 *    (MAX_SPEC_LEN, §12.5.4 of the book chapter).
 *  - Target distribution p_i = softmax(l_t / T_r): temperature applied to the
 *    target only, q used as given ("以小博大" §12.2.3).
 *  - Draft distribution q_i = draft_probs[d], or one-hot at the draft token when
 *    no draft probabilities are given ("以小博大" §12.2.3 and §12.9: draft_probs is
 *    None, the draft is a deterministic proposal).
 *  - Sequentially over i: accept x* = draft_ids[d] iff u_acc * q_i(x*) < p_i(x*),
 *    i.e. with probability min(1, p/q) ("以小博大" §12.2.1; the division-free
 *    "coin * q < p" form of "投机解码端到端深挖" §7.3).  Stop at the first
 *    rejection: later drafts are discarded ("vllm v1 源码精读（五）" §7,
 *    "投机解码端到端深挖" §7 common rules).
 *  - At the first rejected position j: sample the recovered token from
 *    p'(x) = max(0, p(x) - q(x)) / sum_y max(0, p(y) - q(y)) ("以小博大" §12.2.1);
 *    with one-hot q that residual is p with p(x*) set to zero ("以小博大" §12.9).
 *    If every draft is accepted, sample the bonus token from p at position k
 *    ("以小博大" §12.3.2; "投机解码端到端深挖" §7.4, §8.3).
 *  - Temperature 0 (here: T_r <= 0, which also covers the -1 greedy sentinel of
 *    "以小博大" §12.9): accept iff x* equals the target argmax; the output at j is
 *    the target argmax at j ("以小博大" §12.2.4; "投机解码端到端深挖" §7.1).
 *
 * Readings where the pages leave a step open (all listed in the design notes):
 *  - sampling is by inverse CDF in ascending token order: emit the smallest v
 *    with C(v) > theta, theta = u_s * Z, C the inclusive prefix sum of the
 *    residual and Z its total; if rounding leaves theta >= C(V-1), emit the last
 *    v with positive residual mass;
 *  - argmax ties go to the lowest index;
 *  - two uniforms per target row: column 0 is the acceptance coin, column 1 the
 *    sampling draw (used only at the output row);
 *  - an empty residual (Z <= 0, reachable only through rounding or q(x*) = 0)
 *    falls back to sampling p itself, and is flagged;
 *  - out_num_accepted counts accepted drafts only; the recovered / bonus token
 *    is not counted ("投机解码端到端深挖" §8.1: accept_lens = correct + 1);
 *  - rows after the output row are padded with -1.
 *
 * Arithmetic: every probability is formed in double precision from the logits
 * widened exactly (fp32 -> double, bf16 -> fp32 -> double), with libm exp and
 * sums in ascending index order.  There is no blocking, fusion or reordering.
 *
 * Beside each request's result the oracle reports how close each decision it
 * took came to a boundary, so that a lower-precision implementation can be
 * compared draw by draw (the flags below).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_SPEC_LEN 32

/* Per-request flags. */
#define OF_NEAR_ACCEPT 1u      /* |u*q* - p*| <= 1e-5 * max(p*, u*q*) at a visited position  */
#define OF_NEAR_SAMPLE 2u      /* theta within 1e-5 * Z of a CDF boundary at the output row   */
#define OF_NEAR_SAMPLE_ABS 4u  /* explicit-q residual row: theta within 2e-6 of a boundary   */
#define OF_DEGENERATE 8u       /* residual mass Z <= 0: sampled p itself                      */
#define OF_BAD_INPUT 16u       /* request rejected as invalid: out_num_accepted = -1          */
#define OF_NONFINITE 32u       /* a visited row had NaN / +inf / an all -inf maximum          */
#define OF_NEAR_TOPP 64u       /* a top-p cut: the cumulative mass within 5e-6 of top_p       */

#define REL_BAND 1e-5
#define ABS_BAND 2e-6
#define TOPP_BAND 5e-6 /* relative band of the top-p cut (single tokens can carry ~1e-5 of the mass) */

typedef struct {
    const void *logits;
    int dtype; /* 0 = fp32, 1 = bf16 (raw uint16 bits) */
    int64_t T;
    int32_t V;
    int64_t row_stride; /* elements between consecutive target rows */
} logit_rows;

static double logit_at(const logit_rows *L, int64_t t, int32_t v)
{
    if (L->dtype == 0)
        return (double)((const float *)L->logits)[t * L->row_stride + v];
    uint32_t bits = (uint32_t)((const uint16_t *)L->logits)[t * L->row_stride + v] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Largest logit of row t; *nonfinite set if a NaN or +inf is present or the maximum is -inf. */
static double row_max(const logit_rows *L, int64_t t, int *nonfinite)
{
    double m = -INFINITY;
    int bad = 0;
    for (int32_t v = 0; v < L->V; ++v) {
        double l = logit_at(L, t, v);
        if (isnan(l) || l == INFINITY)
            bad = 1;
        if (l > m)
            m = l;
    }
    if (m == -INFINITY)
        bad = 1;
    if (nonfinite)
        *nonfinite = bad;
    return m;
}

/* Lowest index attaining the largest logit, compared on the raw values (no rounding involved). */
static int32_t row_argmax(const logit_rows *L, int64_t t)
{
    int32_t best = 0;
    double bv = logit_at(L, t, 0);
    for (int32_t v = 1; v < L->V; ++v) {
        double l = logit_at(L, t, v);
        if (l > bv) {
            bv = l;
            best = v;
        }
    }
    return best;
}

/* Optional top-k / top-p restriction of the target distribution ("以小博大" §12.2.3, §12.9:
 * the target gets temperature, then top-k / top-p).  top_k <= 0 or >= V and top_p >= 1 (or
 * <= 0) mean "off". */
typedef struct {
    int32_t top_k;
    double top_p;
    double *scratch; /* V doubles, for sorting */
} filter_spec;

static int cmp_desc(const void *a, const void *b)
{
    double x = *(const double *)a, y = *(const double *)b;
    return (x < y) - (x > y);
}

/*
 * p(v) = exp((l(v) - m) / temp) / S over the kept tokens (0 elsewhere), S their total.
 * Kept: all tokens without a filter; with top-k the tokens whose logit is at least the
 * k-th largest logit (ties kept); with top-p, among those, the tokens whose logit is at
 * least that of the token at which the descending cumulative probability first reaches
 * top_p (ties kept).  Returns S; lowers *topp_margin to the relative distance between
 * top_p and the cumulative on either side of the cut.
 */
static double row_softmax_f(const logit_rows *L, int64_t t, double temp, const filter_spec *F, double *p,
                            double *m_out, int *nonfinite, double *topp_margin)
{
    const int32_t V = L->V;
    double m = row_max(L, t, nonfinite);
    double cut = -INFINITY;
    const int use_k = F && F->top_k > 0 && F->top_k < V;
    const int use_p = F && F->top_p > 0.0 && F->top_p < 1.0;
    if (use_k || use_p) {
        double *sorted = F->scratch;
        for (int32_t v = 0; v < V; ++v)
            sorted[v] = logit_at(L, t, v);
        qsort(sorted, (size_t)V, sizeof(double), cmp_desc);
        if (use_k)
            cut = sorted[F->top_k - 1];
        if (use_p) {
            double Sk = 0.0;
            for (int32_t i = 0; i < V && sorted[i] >= cut; ++i)
                Sk += exp((sorted[i] - m) / temp);
            double cum = 0.0;
            for (int32_t i = 0; i < V && sorted[i] >= cut; ++i) {
                double before = cum;
                cum += exp((sorted[i] - m) / temp) / Sk;
                if (cum >= F->top_p) {
                    if (topp_margin) {
                        const double d1 = fabs(cum - F->top_p) / F->top_p, d2 = fabs(before - F->top_p) / F->top_p;
                        const double d = d1 < d2 ? d1 : d2;
                        if (d < *topp_margin)
                            *topp_margin = d;
                    }
                    if (sorted[i] > cut)
                        cut = sorted[i];
                    break;
                }
            }
        }
    }
    double S = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        const double l = logit_at(L, t, v);
        p[v] = (l >= cut) ? exp((l - m) / temp) : 0.0;
        S += p[v];
    }
    for (int32_t v = 0; v < V; ++v)
        p[v] /= S;
    if (m_out)
        *m_out = m;
    return S;
}

/* p(v) = exp((l(v) - m) / temp) / S with S = sum_v exp((l(v) - m) / temp). Returns S. */
static double row_softmax(const logit_rows *L, int64_t t, double temp, double *p, double *m_out, int *nonfinite)
{
    return row_softmax_f(L, t, temp, NULL, p, m_out, nonfinite, NULL);
}

/*
 * Inverse-CDF draw from the (unnormalised) mass r[0..V-1] with total Z:
 * smallest v with C(v) > theta, theta = u * Z.  Sets *margin to the distance
 * from theta to the nearest boundary of the chosen interval.
 */
static int32_t inverse_cdf(const double *r, int32_t V, double Z, double u, double *margin)
{
    double theta = u * Z;
    double C = 0.0, Cprev = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        Cprev = C;
        C += r[v];
        if (C > theta) {
            double a = theta - Cprev, b = C - theta;
            *margin = a < b ? a : b;
            return v;
        }
    }
    /* Rounding left theta at or beyond the total: take the last token with mass. */
    for (int32_t v = V - 1; v >= 0; --v) {
        if (r[v] > 0.0) {
            *margin = 0.0;
            return v;
        }
    }
    *margin = 0.0;
    return V - 1;
}

/*
 * The oracle.  Argument meaning and layout are those of the library's
 * spec_reject_sample, with host pointers, plus:
 *   q_row_stride      elements between draft-probability rows (0 = every row aliases row 0)
 *   out_flags[B]      per-request OF_* flags (may be NULL)
 *   dbg_row_max[T], dbg_row_sum[T], dbg_row_argmax[T]
 *                     per target row: max logit, S = sum exp((l - m)/T_r) (0 on greedy rows), argmax
 *   dbg_p_draft[T-B]  per draft row: p(x*) (0 on greedy rows or bad ids)
 *   dbg_z[B]          per request: normalised residual mass at the output row (1 for the
 *                     bonus, 0 for greedy)
 *   dbg_margin[3*B]   per request: [0] the smallest relative acceptance margin
 *                     |u*q* - p*| / max(p*, u*q*) over the visited positions, [1] the
 *                     sampling margin (distance from theta to the nearest boundary of
 *                     the chosen interval) divided by Z, [2] the smallest relative
 *                     distance of a top-p cut's cumulative to top_p; +inf where not
 *                     applicable
 *   top_k[B], top_p[B] optional per-request target filters (NULL = off), applied to every
 *                     sampled row of the request (greedy requests ignore them)
 * Every dbg_* pointer may be NULL.  nthreads <= 0 uses the OpenMP default.
 * Returns 0, or 1 when the batch as a whole is inconsistent (cu[0] != 0, cu[B] + B != T or
 * cu decreasing), in which case every request is reported invalid and no token is written.
 */
int oracle_reject_sample(const void *target_logits, int dtype, int64_t T, int32_t V, int64_t logits_row_stride,
                         const float *draft_probs, int64_t q_row_stride, const int32_t *draft_ids,
                         const int32_t *cu_num_draft, int32_t B, const float *uniforms, const float *temperature,
                         int32_t *out_tokens, int32_t *out_num_accepted, uint32_t *out_flags, double *dbg_row_max,
                         double *dbg_row_sum, int32_t *dbg_row_argmax, double *dbg_p_draft, double *dbg_z,
                         double *dbg_margin, int nthreads, const int32_t *top_k, const float *top_p)
{
    logit_rows L = {target_logits, dtype, T, V, logits_row_stride};
    const int64_t num_draft_rows = T - B;
    /* The flattened layout itself is broken when cu does not start at 0, does not
     * end at T - B, or decreases: then no request's rows are known. */
    int global_bad = (B < 0 || V < 1 || cu_num_draft[0] != 0 || (int64_t)cu_num_draft[B] + B != T);
    for (int32_t req = 0; !global_bad && req < B; ++req)
        if (cu_num_draft[req + 1] < cu_num_draft[req])
            global_bad = 1;

#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        double *srt = (double *)malloc(sizeof(double) * (size_t)V);

#pragma omp for schedule(dynamic, 1)
        for (int32_t req = 0; req < B; ++req) {
            uint32_t flags = 0;
            int64_t k = (int64_t)cu_num_draft[req + 1] - cu_num_draft[req];
            int64_t tb = (int64_t)cu_num_draft[req] + req; /* first target row */
            int64_t db = cu_num_draft[req];                /* first draft row  */
            int bad = global_bad || k < 0 || k > ORACLE_MAX_SPEC_LEN || db < 0 || tb + k + 1 > T ||
                      db + k > num_draft_rows;
            for (int64_t i = 0; !bad && i < k; ++i)
                if (draft_ids[db + i] < 0 || draft_ids[db + i] >= V)
                    bad = 1;
            if (bad) {
                /* Too many drafts or a draft id outside [0, V): this request only. */
                out_num_accepted[req] = -1;
                if (!global_bad)
                    for (int64_t i = 0; i <= k; ++i)
                        out_tokens[tb + i] = -1;
                if (out_flags)
                    out_flags[req] = OF_BAD_INPUT;
                if (dbg_z)
                    dbg_z[req] = 0.0;
                continue;
            }

            const double temp = (double)temperature[req];
            const int greedy = !(temp > 0.0);
            const filter_spec F = {top_k ? top_k[req] : 0, top_p ? (double)top_p[req] : 1.0, srt};
            double topp_margin = INFINITY;
            int64_t j = k; /* output position: first rejection, or k for the bonus */
            int nonfinite = 0;
            double margin_accept = INFINITY, margin_sample = INFINITY;

            /* Acceptance test, sequential over the drafts, stopping at the first rejection. */
            for (int64_t i = 0; i < k; ++i) {
                const int64_t t = tb + i, d = db + i;
                const int32_t xs = draft_ids[d];
                if (greedy) {
                    if (xs != row_argmax(&L, t)) {
                        j = i;
                        break;
                    }
                    continue;
                }
                int nf = 0;
                row_softmax_f(&L, t, temp, &F, p, NULL, &nf, &topp_margin);
                nonfinite |= nf;
                const double qs = draft_probs ? (double)draft_probs[d * q_row_stride + xs] : 1.0;
                const double us = (double)uniforms[2 * t + 0];
                const double lhs = us * qs, rhs = p[xs];
                const double big = lhs > rhs ? lhs : rhs;
                if (fabs(lhs - rhs) <= REL_BAND * big)
                    flags |= OF_NEAR_ACCEPT;
                if (big > 0.0 && fabs(lhs - rhs) / big < margin_accept)
                    margin_accept = fabs(lhs - rhs) / big;
                if (!(lhs < rhs)) {
                    j = i;
                    break;
                }
            }

            /* The token at position j: recovered (j < k) or bonus (j == k). */
            const int64_t t = tb + j;
            int32_t token;
            double zr = 0.0;
            if (greedy) {
                token = row_argmax(&L, t);
            } else {
                int nf = 0;
                row_softmax_f(&L, t, temp, &F, p, NULL, &nf, &topp_margin);
                nonfinite |= nf;
                int explicit_residual = 0;
                if (j < k) {
                    const int64_t d = db + j;
                    const int32_t xs = draft_ids[d];
                    if (draft_probs) {
                        const float *q = draft_probs + d * q_row_stride;
                        for (int32_t v = 0; v < V; ++v) {
                            double diff = p[v] - (double)q[v];
                            r[v] = diff > 0.0 ? diff : 0.0;
                        }
                        explicit_residual = 1;
                    } else {
                        for (int32_t v = 0; v < V; ++v)
                            r[v] = p[v];
                        r[xs] = 0.0;
                    }
                } else {
                    for (int32_t v = 0; v < V; ++v)
                        r[v] = p[v];
                }
                double Z = 0.0;
                for (int32_t v = 0; v < V; ++v)
                    Z += r[v];
                const double us = (double)uniforms[2 * t + 1];
                double margin;
                if (Z > 0.0) {
                    zr = Z;
                    token = inverse_cdf(r, V, Z, us, &margin);
                    margin_sample = margin / Z;
                    if (margin <= REL_BAND * Z)
                        flags |= OF_NEAR_SAMPLE;
                    if (explicit_residual && margin <= ABS_BAND)
                        flags |= OF_NEAR_SAMPLE_ABS;
                } else {
                    flags |= OF_DEGENERATE;
                    double Zp = 0.0;
                    for (int32_t v = 0; v < V; ++v)
                        Zp += p[v];
                    token = inverse_cdf(p, V, Zp, us, &margin);
                    margin_sample = margin / Zp;
                    if (margin <= REL_BAND * Zp)
                        flags |= OF_NEAR_SAMPLE;
                }
            }

            for (int64_t i = 0; i < j; ++i)
                out_tokens[tb + i] = draft_ids[db + i];
            out_tokens[t] = token;
            for (int64_t i = j + 1; i <= k; ++i)
                out_tokens[tb + i] = -1;
            out_num_accepted[req] = (int32_t)j;
            if (nonfinite)
                flags |= OF_NONFINITE;
            if (topp_margin <= TOPP_BAND)
                flags |= OF_NEAR_TOPP;
            if (out_flags)
                out_flags[req] = flags;
            if (dbg_z)
                dbg_z[req] = greedy ? 0.0 : zr;
            if (dbg_margin) {
                dbg_margin[3 * req] = margin_accept;
                dbg_margin[3 * req + 1] = margin_sample;
                dbg_margin[3 * req + 2] = topp_margin;
            }
        }

        /* Per-row statistics for every row (debug outputs only). */
        if (!global_bad && (dbg_row_max || dbg_row_sum || dbg_row_argmax || dbg_p_draft)) {
#pragma omp for schedule(dynamic, 1)
            for (int32_t req = 0; req < B; ++req) {
                int64_t k = (int64_t)cu_num_draft[req + 1] - cu_num_draft[req];
                int64_t tb = (int64_t)cu_num_draft[req] + req, db = cu_num_draft[req];
                if (k < 0 || k > ORACLE_MAX_SPEC_LEN || tb + k + 1 > T || db + k > num_draft_rows)
                    continue;
                const double temp = (double)temperature[req];
                const int greedy = !(temp > 0.0);
                const filter_spec F = {top_k ? top_k[req] : 0, top_p ? (double)top_p[req] : 1.0, srt};
                for (int64_t i = 0; i <= k; ++i) {
                    const int64_t t = tb + i;
                    double m, S = 0.0;
                    if (greedy) {
                        m = row_max(&L, t, NULL);
                    } else {
                        S = row_softmax_f(&L, t, temp, &F, p, &m, NULL, NULL);
                    }
                    if (dbg_row_max)
                        dbg_row_max[t] = m;
                    if (dbg_row_sum)
                        dbg_row_sum[t] = S;
                    if (dbg_row_argmax)
                        dbg_row_argmax[t] = row_argmax(&L, t);
                    if (dbg_p_draft && i < k) {
                        const int32_t xs = draft_ids[db + i];
                        dbg_p_draft[db + i] = (greedy || xs < 0 || xs >= V) ? 0.0 : p[xs];
                    }
                }
            }
        }
        free(p);
        free(r);
        free(srt);
    }

    if (global_bad) {
        for (int32_t req = 0; req < B; ++req) {
            out_num_accepted[req] = -1;
            if (out_flags)
                out_flags[req] = OF_BAD_INPUT;
        }
        return 1;
    }
    return 0;
}

/* Number of OpenMP threads the oracle would use (1 when built without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
