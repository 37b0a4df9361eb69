/*
 * spec_ref.c -- plain, slow, fp64 CPU oracle for batched speculative-sampling
 * verification.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline / reference arm load this library.  The CUDA product path never
 * calls, links or includes anything here, and this file includes nothing from
 * the product (no shared headers, tables or helpers).
 *
 * What it computes, and where the pages define it:
 *   - p = softmax(logits / T), q likewise, same T for target and draft:
 *     "Speculative Decoding and the Art of Fast LLM Inference", "Why It Stays
 *     Exact", key limitation (identical temperature for draft and target).
 *   - accept g_i with probability min(1, p_i(g_i)/q_i(g_i)), left to right:
 *     same page, "The Algorithm, Step by Step", step "Accept or reject";
 *     "Speculative decoding: faster LLM inference" (thelatentsource),
 *     "The correction that keeps the target in charge", the accept_token
 *     snippet: draft_prob <= 0 is an error, target_prob >= draft_prob accepts,
 *     otherwise accept iff a uniform in [0,1) is strictly below the ratio.
 *   - stop at the first rejection and draw one token from
 *     norm(max(0, p - q)) there: first page, step "Stop at the first
 *     rejection"; second page, equation r(x).
 *   - if all k are accepted, draw a bonus token from p_{k+1}: first page, step
 *     "Bonus token"; interview page ("techaiinterview"), "Algorithm (one
 *     round)", step 4.
 *   - temperature 0: accept while the target's argmax equals the draft token:
 *     interview page, "Deep dive: correctness and speedup" (greedy remark).
 *
 * Readings where the pages are silent (taken as the plainest reading the rest
 * of the pages supports):
 *   - a draw uses inverse-CDF: C(x) = sum_{y<=x} w(y) accumulated left to
 *     right, R = C(V-1) (the scan's own total), token = smallest x with
 *     C(x) > u*R; if rounding leaves no such x, the largest x with w(x) > 0.
 *   - u_accept[b,i] drives accept test i; u_resample[b] drives the one draw.
 *   - residual mass R == 0 at a rejection (impossible in exact arithmetic)
 *     falls back to sampling p_j.
 *   - argmax ties go to the lowest index.
 *   - sequence errors (out_num_accepted = -1, tokens all -1): T NaN, negative,
 *     infinite, or positive below FLT_MIN; a draft token outside [0,V); a NaN
 *     or +inf logit in a row the call reads (all k+1 target rows, and the k
 *     draft rows when T > 0); such a row whose logits are all -inf; q(g) <= 0
 *     at a position the scan reaches.
 *
 * Sampling (spec_sample_ref): the draft model's step before verification,
 * each proposed token sampled from its distribution q ("Speculative Decoding
 * and the Art of Fast LLM Inference", "The Algorithm, Step by Step", the
 * drafting step; interview page, "Algorithm (one round)", step 1).  One token
 * per row: T > 0 draws from softmax(l / T) by the same inverse-CDF reading as
 * the verification's draws; T == 0 takes the argmax (lowest index on ties);
 * row errors (token -1): T invalid as above, a NaN or +inf logit, or every
 * logit -inf.
 *
 * Tree verification (spec_verify_tree_ref_mt): several candidate
 * continuations per sequence; the reading of its sibling rule is stated
 * above that function.
 *
 * Everything is fp64 with plain sequential loops; no blocking, no fusion, no
 * reordering beyond the definition.
 */
#define _GNU_SOURCE /* qsort_r */
#include <math.h>
#include <float.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

#define REF_F32 0
#define REF_BF16 1

#define REF_OK 0
#define REF_EINVAL 1
#define REF_ENOMEM 2

/* ---------------------------------------------------------------- decoding */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double ref_bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Read one logit of a row-major array as fp64. */
static double ref_logit(const void *base, int dtype, size_t idx)
{
    if (dtype == REF_F32)
        return (double)((const float *)base)[idx];
    return ref_bf16_to_double(((const uint16_t *)base)[idx]);
}

/* Copy row `row` (V logits) of a typed array into an fp64 buffer. */
static void ref_load_row(const void *base, int dtype, size_t row, int64_t V, double *out)
{
    for (int64_t x = 0; x < V; ++x)
        out[x] = ref_logit(base, dtype, (size_t)row * (size_t)V + (size_t)x);
}

/* ------------------------------------------------------------- primitives */

/* Maximum and lowest-index argmax of a row. */
static double ref_max_argmax(const double *l, int64_t V, int64_t *arg)
{
    double m = l[0];
    int64_t a = 0;
    for (int64_t x = 1; x < V; ++x) {
        if (l[x] > m) {
            m = l[x];
            a = x;
        }
    }
    if (arg)
        *arg = a;
    return m;
}

/* 1 if the row holds a NaN or +inf, or every entry is -inf. */
static int ref_row_invalid(const double *l, int64_t V)
{
    int all_neg_inf = 1;
    for (int64_t x = 0; x < V; ++x) {
        if (isnan(l[x]) || (isinf(l[x]) && l[x] > 0))
            return 1;
        if (!(isinf(l[x]) && l[x] < 0))
            all_neg_inf = 0;
    }
    return all_neg_inf;
}

/*
 * p = softmax(l / T) over V entries, T > 0, with the maximum subtracted
 * before exponentiation (exp(-inf) = 0 for masked entries).
 */
int spec_ref_softmax(const double *l, int64_t V, double T, double *p)
{
    if (!(T > 0) || V < 1)
        return REF_EINVAL;
    double m = ref_max_argmax(l, V, NULL);
    double Z = 0.0;
    for (int64_t x = 0; x < V; ++x) {
        p[x] = exp((l[x] - m) / T);
        Z += p[x];
    }
    for (int64_t x = 0; x < V; ++x)
        p[x] /= Z;
    return REF_OK;
}

/* Order of a sort by logit descending, index ascending (keys in `arg`). */
static int ref_order_cmp(const void *a, const void *b, void *arg)
{
    const double *l = (const double *)arg;
    const int64_t i = *(const int64_t *)a, j = *(const int64_t *)b;
    if (l[i] > l[j])
        return -1;
    if (l[i] < l[j])
        return 1;
    return (i < j) ? -1 : (i > j);
}

/*
 * Top-k / top-p filtered softmax.  Tokens are ranked by logit, descending,
 * ties by index ascending.  top-k keeps the first K of them (K <= 0 or
 * K >= V: all).  top-p keeps, among those, a token while the mass ranked
 * strictly before it is below P * Z_K, Z_K the mass of the top-k set (P >= 1:
 * all of them); at least one token is always kept.  p receives the
 * distribution renormalised over the kept set (0 elsewhere).  *margin (if
 * non-NULL) receives the distance of the two decisive running masses from
 * P * Z_K, relative to Z_K (NaN without top-p).  Returns the kept count, or
 * -1 on bad arguments.
 */
int64_t spec_ref_filtered_softmax(const double *l, int64_t V, double T, int64_t K, double P,
                                  double *p, double *margin)
{
    if (!(T > 0) || V < 1)
        return -1;
    int64_t *order = (int64_t *)malloc((size_t)V * sizeof(int64_t));
    double *e = (double *)malloc((size_t)V * sizeof(double));
    if (!order || !e) {
        free(order);
        free(e);
        return -1;
    }
    double m = ref_max_argmax(l, V, NULL);
    for (int64_t x = 0; x < V; ++x) {
        e[x] = exp((l[x] - m) / T);
        order[x] = x;
    }
    qsort_r(order, (size_t)V, sizeof(int64_t), ref_order_cmp, (void *)l);
    const int64_t Keff = (K > 0 && K < V) ? K : V;
    double ZK = 0.0;
    for (int64_t i = 0; i < Keff; ++i)
        ZK += e[order[i]];
    int64_t N = Keff;
    double mg = NAN;
    if (P < 1.0) {
        const double target = P * ZK;
        double cum = 0.0, before_last = 0.0;
        for (int64_t i = 0; i < Keff; ++i) {
            if (cum >= target) {
                N = i;
                break;
            }
            before_last = cum;
            cum += e[order[i]];
        }
        /* decisive comparisons: the last kept token (before < target) and,
           if any token was cut, the first cut one (before >= target) */
        mg = (target - before_last) / ZK;
        if (N < Keff) {
            const double m2 = (cum - target) / ZK;
            if (m2 < mg)
                mg = m2;
        }
    }
    double Z = 0.0;
    for (int64_t x = 0; x < V; ++x)
        p[x] = 0.0;
    for (int64_t i = 0; i < N; ++i) {
        p[order[i]] = e[order[i]];
        Z += e[order[i]];
    }
    for (int64_t i = 0; i < N; ++i)
        p[order[i]] /= Z;
    if (margin)
        *margin = mg;
    free(order);
    free(e);
    return N;
}

/*
 * Residual (correction) weights w(x) = max(0, p(x) - q(x)); returns their
 * total.  The normalised r(x) = w(x) / total is the second page's r(x).
 */
double spec_ref_residual(const double *p, const double *q, int64_t V, double *w)
{
    double R = 0.0;
    for (int64_t x = 0; x < V; ++x) {
        double d = p[x] - q[x];
        w[x] = d > 0.0 ? d : 0.0;
        R += w[x];
    }
    return R;
}

/*
 * Inverse-CDF draw from non-negative weights w (not necessarily normalised):
 * C(x) = sum_{y<=x} w(y), R = C(V-1); the smallest x with C(x) > u*R, else
 * the largest x with w(x) > 0.  Returns -1 if every weight is zero.  When
 * cell is non-NULL it receives [C(x-1)/R, C(x)/R, R] for the chosen x.
 */
int64_t spec_ref_inverse_cdf(const double *w, int64_t V, double u, double *cell)
{
    double R = 0.0;
    for (int64_t x = 0; x < V; ++x)
        R += w[x];
    if (!(R > 0.0))
        return -1;
    double target = u * R;
    double C = 0.0, Cprev = 0.0;
    int64_t pick = -1;
    for (int64_t x = 0; x < V; ++x) {
        Cprev = C;
        C += w[x];
        if (C > target) {
            pick = x;
            break;
        }
    }
    if (pick < 0) {
        /* rounding left u*R at or above the total: clamp */
        for (int64_t x = V - 1; x >= 0; --x) {
            if (w[x] > 0.0) {
                pick = x;
                break;
            }
        }
        C = 0.0;
        for (int64_t x = 0; x <= pick; ++x) {
            Cprev = C;
            C += w[x];
        }
    }
    if (cell) {
        cell[0] = Cprev / R;
        cell[1] = C / R;
        cell[2] = R;
    }
    return pick;
}

/* ------------------------------------------------------------ one sequence */

typedef struct {
    const void *target;      /* [B, k+1, V] */
    const void *draft;       /* [B, k, V] */
    int dtype;
    const int32_t *tokens;   /* [B, k] */
    const double *u_accept;  /* [B, k] */
    const double *u_resample;/* [B] */
    const double *temperature;/* [B] */
    int64_t B, k, V;
    int32_t *out_tokens;     /* [B, k+1] */
    int32_t *out_num_accepted;/* [B] */
    double *trace;           /* [B, tw] or NULL */
    int64_t tw;              /* trace width: k+3, or k+4 with the filter margin */
    const int32_t *top_k;    /* [B] or NULL (no top-k) */
    const double *top_p;     /* [B] or NULL (no top-p) */
    int64_t b0, b1;          /* sequence range for this worker */
    int status;
} ref_job_t;

/* The sequence's sampling distribution of one row: softmax(l/T), filtered by
   the sequence's top-k / top-p when the call has them; tracks the smallest
   top-p margin seen. */
static void ref_dist(const ref_job_t *J, int64_t b, const double *l, double T, double *p,
                     double *min_margin)
{
    const int64_t K = J->top_k ? J->top_k[b] : 0;
    const double P = J->top_p ? J->top_p[b] : 1.0;
    if ((K <= 0 || K >= J->V) && !(P < 1.0)) {  /* no filter at all */
        spec_ref_softmax(l, J->V, T, p);
        return;
    }
    double mg = NAN;
    spec_ref_filtered_softmax(l, J->V, T, K, P, p, &mg);
    if (!isnan(mg) && (isnan(*min_margin) || mg < *min_margin))
        *min_margin = mg;
}

static void ref_fail_sequence(ref_job_t *J, int64_t b)
{
    for (int64_t i = 0; i <= J->k; ++i)
        J->out_tokens[b * (J->k + 1) + i] = -1;
    J->out_num_accepted[b] = -1;
}

/* Returns 0 on success, 1 if the sequence is an error row. */
static int ref_one_sequence(ref_job_t *J, int64_t b, double *t, double *d,
                            double *p, double *q, double *w)
{
    const int64_t k = J->k, V = J->V;
    const double T = J->temperature[b];
    double *tr = J->trace ? J->trace + b * J->tw : NULL;
    if (tr)
        for (int64_t i = 0; i < J->tw; ++i)
            tr[i] = NAN;
    double min_margin = NAN;

    /* temperature must be 0 (greedy) or a finite normal positive value */
    if (isnan(T) || T < 0 || isinf(T) || (T > 0 && T < (double)FLT_MIN))
        return 1;
    /* filter parameters: top-k >= 0, top-p in (0, 1] or above (no top-p) */
    if (J->top_k && J->top_k[b] < 0)
        return 1;
    if (J->top_p && (isnan(J->top_p[b]) || !(J->top_p[b] > 0.0)))
        return 1;
    for (int64_t i = 0; i < k; ++i) {
        int32_t g = J->tokens[b * k + i];
        if (g < 0 || g >= V)
            return 1;
    }
    /* every row the call reads must be usable */
    for (int64_t i = 0; i <= k; ++i) {
        ref_load_row(J->target, J->dtype, (size_t)(b * (k + 1) + i), V, t);
        if (ref_row_invalid(t, V))
            return 1;
    }
    if (T > 0) {
        for (int64_t i = 0; i < k; ++i) {
            ref_load_row(J->draft, J->dtype, (size_t)(b * k + i), V, d);
            if (ref_row_invalid(d, V))
                return 1;
        }
    }

    int64_t j = k;        /* first rejected position, k = all accepted */
    int64_t token = -1;
    if (T == 0) {
        /* greedy: accept while the target's argmax equals the draft token */
        for (int64_t i = 0; i < k; ++i) {
            int64_t a;
            ref_load_row(J->target, J->dtype, (size_t)(b * (k + 1) + i), V, t);
            ref_max_argmax(t, V, &a);
            if (J->tokens[b * k + i] != a) {
                j = i;
                token = a;
                break;
            }
        }
        if (j == k) {
            int64_t a;
            ref_load_row(J->target, J->dtype, (size_t)(b * (k + 1) + k), V, t);
            ref_max_argmax(t, V, &a);
            token = a;
        }
    } else {
        for (int64_t i = 0; i < k; ++i) {
            int32_t g = J->tokens[b * k + i];
            ref_load_row(J->target, J->dtype, (size_t)(b * (k + 1) + i), V, t);
            ref_load_row(J->draft, J->dtype, (size_t)(b * k + i), V, d);
            ref_dist(J, b, t, T, p, &min_margin);
            ref_dist(J, b, d, T, q, &min_margin);
            double P = p[g], Q = q[g];
            if (Q <= 0.0)
                return 1; /* a sampled draft token must have positive probability */
            double ratio = P / Q;
            if (tr)
                tr[i] = ratio < 1.0 ? ratio : 1.0;
            int accept = (P >= Q) || (J->u_accept[b * k + i] < ratio);
            if (!accept) {
                j = i;
                break;
            }
        }
        double cell[3];
        if (j < k) {
            /* p and q still hold position j's distributions */
            double R = spec_ref_residual(p, q, V, w);
            if (!(R > 0.0))
                memcpy(w, p, (size_t)V * sizeof(double)); /* rounding-only fallback */
        } else {
            ref_load_row(J->target, J->dtype, (size_t)(b * (k + 1) + k), V, t);
            ref_dist(J, b, t, T, w, &min_margin);
        }
        token = spec_ref_inverse_cdf(w, V, J->u_resample[b], cell);
        if (token < 0)
            return 1;
        if (tr) {
            tr[k] = cell[0];
            tr[k + 1] = cell[1];
            tr[k + 2] = cell[2];
            if (J->tw > k + 3)
                tr[k + 3] = min_margin;
        }
    }

    for (int64_t i = 0; i < j; ++i)
        J->out_tokens[b * (k + 1) + i] = J->tokens[b * k + i];
    J->out_tokens[b * (k + 1) + j] = (int32_t)token;
    for (int64_t i = j + 1; i <= k; ++i)
        J->out_tokens[b * (k + 1) + i] = -1;
    J->out_num_accepted[b] = (int32_t)j;
    return 0;
}

static void *ref_worker(void *arg)
{
    ref_job_t *J = (ref_job_t *)arg;
    size_t n = (size_t)J->V;
    double *buf = (double *)malloc(5 * n * sizeof(double));
    if (!buf) {
        J->status = REF_ENOMEM;
        return NULL;
    }
    double *t = buf, *d = buf + n, *p = buf + 2 * n, *q = buf + 3 * n, *w = buf + 4 * n;
    for (int64_t b = J->b0; b < J->b1; ++b)
        if (ref_one_sequence(J, b, t, d, p, q, w))
            ref_fail_sequence(J, b);
    free(buf);
    J->status = REF_OK;
    return NULL;
}

/*
 * The verification step for B sequences, split over `nthreads` host threads
 * (contiguous ranges of sequences; the result does not depend on the split).
 *
 * target [B,k+1,V] and draft [B,k,V] are fp32 or bf16 bit patterns (dtype 0
 * or 1).  Uniforms and temperatures are fp64 so that tests can place them
 * anywhere in [0,1).  trace (nullable) receives per sequence k+3 doubles: the
 * accept threshold min(1, P/Q) of each tested position (NaN if not tested or
 * greedy), then the chosen draw cell [lo, hi) in u-units and the draw's total
 * mass R (NaN for greedy).
 */
static int ref_verify_core(const void *target, const void *draft, int dtype,
                           const int32_t *tokens, const double *u_accept,
                           const double *u_resample, const double *temperature,
                           const int32_t *top_k, const double *top_p, int filtered,
                           int64_t B, int64_t k, int64_t V,
                           int32_t *out_tokens, int32_t *out_num_accepted,
                           double *trace, int nthreads);

int spec_verify_ref_mt(const void *target, const void *draft, int dtype,
                       const int32_t *tokens, const double *u_accept,
                       const double *u_resample, const double *temperature,
                       int64_t B, int64_t k, int64_t V,
                       int32_t *out_tokens, int32_t *out_num_accepted,
                       double *trace, int nthreads)
{
    return ref_verify_core(target, draft, dtype, tokens, u_accept, u_resample, temperature,
                           NULL, NULL, 0, B, k, V, out_tokens, out_num_accepted, trace,
                           nthreads);
}

/*
 * The verification step with top-k / top-p filtered distributions
 * (spec_ref_filtered_softmax) for every row of a sequence at T > 0, the same
 * parameters for target and draft.  top_k [B] (0: none; < 0: sequence error)
 * and top_p [B] (>= 1: none; NaN or <= 0: sequence error) may each be NULL.
 * trace (nullable) is [B, k+4]: the k+3 columns of spec_verify_ref_mt and the
 * smallest top-p margin over the rows the sequence read (NaN if none).
 */
int spec_verify_ref_filtered_mt(const void *target, const void *draft, int dtype,
                                const int32_t *tokens, const double *u_accept,
                                const double *u_resample, const double *temperature,
                                const int32_t *top_k, const double *top_p,
                                int64_t B, int64_t k, int64_t V,
                                int32_t *out_tokens, int32_t *out_num_accepted,
                                double *trace, int nthreads)
{
    return ref_verify_core(target, draft, dtype, tokens, u_accept, u_resample, temperature,
                           top_k, top_p, 1, B, k, V, out_tokens, out_num_accepted, trace,
                           nthreads);
}

static int ref_verify_core(const void *target, const void *draft, int dtype,
                           const int32_t *tokens, const double *u_accept,
                           const double *u_resample, const double *temperature,
                           const int32_t *top_k, const double *top_p, int filtered,
                           int64_t B, int64_t k, int64_t V,
                           int32_t *out_tokens, int32_t *out_num_accepted,
                           double *trace, int nthreads)
{
    if (!target || !tokens || !u_accept || !u_resample || !temperature ||
        !out_tokens || !out_num_accepted)
        return REF_EINVAL;
    if (B < 0 || k < 1 || V < 2 || (dtype != REF_F32 && dtype != REF_BF16))
        return REF_EINVAL;
    if (!draft)
        return REF_EINVAL;
    if (B == 0)
        return REF_OK;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > B)
        nthreads = (int)B;

    ref_job_t *jobs = (ref_job_t *)calloc((size_t)nthreads, sizeof(ref_job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return REF_ENOMEM;
    }
    for (int w = 0; w < nthreads; ++w) {
        ref_job_t *J = &jobs[w];
        J->target = target;
        J->draft = draft;
        J->dtype = dtype;
        J->tokens = tokens;
        J->u_accept = u_accept;
        J->u_resample = u_resample;
        J->temperature = temperature;
        J->B = B;
        J->k = k;
        J->V = V;
        J->out_tokens = out_tokens;
        J->out_num_accepted = out_num_accepted;
        J->trace = trace;
        J->tw = filtered ? k + 4 : k + 3;
        J->top_k = top_k;
        J->top_p = top_p;
        J->b0 = B * w / nthreads;
        J->b1 = B * (w + 1) / nthreads;
    }
    int status = REF_OK;
    if (nthreads == 1) {
        ref_worker(&jobs[0]);
        status = jobs[0].status;
    } else {
        int started = 0;
        for (int w = 0; w < nthreads; ++w) {
            if (pthread_create(&th[w], NULL, ref_worker, &jobs[w]) != 0)
                break;
            ++started;
        }
        for (int w = 0; w < started; ++w)
            pthread_join(th[w], NULL);
        for (int w = started; w < nthreads; ++w)
            ref_worker(&jobs[w]);
        for (int w = 0; w < nthreads; ++w)
            if (jobs[w].status != REF_OK)
                status = jobs[w].status;
    }
    free(jobs);
    free(th);
    return status;
}

int spec_verify_ref(const void *target, const void *draft, int dtype,
                    const int32_t *tokens, const double *u_accept,
                    const double *u_resample, const double *temperature,
                    int64_t B, int64_t k, int64_t V,
                    int32_t *out_tokens, int32_t *out_num_accepted, double *trace)
{
    return spec_verify_ref_mt(target, draft, dtype, tokens, u_accept, u_resample,
                              temperature, B, k, V, out_tokens, out_num_accepted,
                              trace, 1);
}

/*
 * Intermediate probabilities P = p_i(g_i) and Q = q_i(g_i) at every draft
 * position (not only the tested ones), out[B,k,2].  Greedy sequences and
 * error rows get NaN.
 */
int spec_ref_probs(const void *target, const void *draft, int dtype,
                   const int32_t *tokens, const double *temperature,
                   int64_t B, int64_t k, int64_t V, double *out)
{
    if (!target || !draft || !tokens || !temperature || !out || V < 2 || k < 1)
        return REF_EINVAL;
    double *buf = (double *)malloc(3 * (size_t)V * sizeof(double));
    if (!buf)
        return REF_ENOMEM;
    double *l = buf, *p = buf + V, *q = buf + 2 * V;
    for (int64_t b = 0; b < B; ++b) {
        double T = temperature[b];
        for (int64_t i = 0; i < k; ++i) {
            double *o = out + (b * k + i) * 2;
            o[0] = o[1] = NAN;
            int32_t g = tokens[b * k + i];
            if (!(T > 0) || isinf(T) || g < 0 || g >= V)
                continue;
            ref_load_row(target, dtype, (size_t)(b * (k + 1) + i), V, l);
            if (ref_row_invalid(l, V))
                continue;
            spec_ref_softmax(l, V, T, p);
            ref_load_row(draft, dtype, (size_t)(b * k + i), V, l);
            if (ref_row_invalid(l, V))
                continue;
            spec_ref_softmax(l, V, T, q);
            o[0] = p[g];
            o[1] = q[g];
        }
    }
    free(buf);
    return REF_OK;
}

/* ----------------------------------------------------------------- sampling */

typedef struct {
    const void *logits;       /* [R, V] */
    int dtype;
    const double *u;          /* [R] */
    const double *temperature;/* [R] */
    int64_t V;
    int32_t *out;             /* [R] */
    double *trace;            /* [R, 3] or NULL */
    int64_t r0, r1;
    int status;
} ref_sample_job_t;

/* One row: returns the token, or -1 on a row error. */
static int64_t ref_sample_row(const ref_sample_job_t *J, int64_t r, double *l, double *p,
                              double *tr)
{
    const int64_t V = J->V;
    const double T = J->temperature[r];
    if (isnan(T) || T < 0 || isinf(T) || (T > 0 && T < (double)FLT_MIN))
        return -1;
    ref_load_row(J->logits, J->dtype, (size_t)r, V, l);
    if (ref_row_invalid(l, V))
        return -1;
    if (T == 0) {
        int64_t a;
        ref_max_argmax(l, V, &a);
        return a;
    }
    spec_ref_softmax(l, V, T, p);
    double cell[3];
    int64_t tok = spec_ref_inverse_cdf(p, V, J->u[r], cell);
    if (tok >= 0 && tr) {
        tr[0] = cell[0];
        tr[1] = cell[1];
        tr[2] = cell[2];
    }
    return tok;
}

static void *ref_sample_worker(void *arg)
{
    ref_sample_job_t *J = (ref_sample_job_t *)arg;
    double *buf = (double *)malloc(2 * (size_t)J->V * sizeof(double));
    if (!buf) {
        J->status = REF_ENOMEM;
        return NULL;
    }
    for (int64_t r = J->r0; r < J->r1; ++r) {
        double *tr = J->trace ? J->trace + r * 3 : NULL;
        if (tr)
            tr[0] = tr[1] = tr[2] = NAN;
        J->out[r] = (int32_t)ref_sample_row(J, r, buf, buf + J->V, tr);
    }
    free(buf);
    J->status = REF_OK;
    return NULL;
}

/*
 * One token per row of logits [R, V] (fp32 or bf16 bit patterns), split over
 * `nthreads` host threads (contiguous row ranges; the result does not depend
 * on the split).  trace (nullable) receives per row the chosen draw cell
 * [C(x-1)/R, C(x)/R) and the total R (NaN for greedy or error rows).
 */
int spec_sample_ref_mt(const void *logits, int dtype, const double *u,
                       const double *temperature, int64_t R, int64_t V,
                       int32_t *out_tokens, double *trace, int nthreads)
{
    if (!logits || !u || !temperature || !out_tokens)
        return REF_EINVAL;
    if (R < 0 || V < 2 || (dtype != REF_F32 && dtype != REF_BF16))
        return REF_EINVAL;
    if (R == 0)
        return REF_OK;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > R)
        nthreads = (int)R;
    ref_sample_job_t *jobs = (ref_sample_job_t *)calloc((size_t)nthreads, sizeof *jobs);
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return REF_ENOMEM;
    }
    for (int w = 0; w < nthreads; ++w) {
        ref_sample_job_t *J = &jobs[w];
        J->logits = logits;
        J->dtype = dtype;
        J->u = u;
        J->temperature = temperature;
        J->V = V;
        J->out = out_tokens;
        J->trace = trace;
        J->r0 = R * w / nthreads;
        J->r1 = R * (w + 1) / nthreads;
    }
    int started = 0;
    if (nthreads > 1)
        for (int w = 0; w < nthreads; ++w) {
            if (pthread_create(&th[w], NULL, ref_sample_worker, &jobs[w]) != 0)
                break;
            ++started;
        }
    for (int w = 0; w < started; ++w)
        pthread_join(th[w], NULL);
    for (int w = started; w < nthreads; ++w)
        ref_sample_worker(&jobs[w]);
    int status = REF_OK;
    for (int w = 0; w < nthreads; ++w)
        if (jobs[w].status != REF_OK)
            status = jobs[w].status;
    free(jobs);
    free(th);
    return status;
}

/* ------------------------------------------------------- tree verification */

/*
 * Tree verification: several candidate continuations per sequence, verified
 * together ("Speculative Decoding and the Art of Fast LLM Inference", "Where
 * the Draft Comes From", "EAGLE: drafting in feature space", on EAGLE-2/3;
 * techaiinterview, "Drafts and limits", the tree-verification line).  The
 * pages name the idea but give no rule for choosing among siblings; the
 * thelatentsource page ("Choosing who does the drafting", on Medusa) warns
 * that tree acceptance variants need not preserve the target distribution.
 * The reading taken here is the one that keeps the exactness argument of the
 * first page ("Why It Stays Exact") node by node:
 *
 *   - node 0 is the root (the last committed position); node n >= 1 holds
 *     draft token tokens[n] and hangs below parent[n] < n.  Target row n is
 *     the target's logits after the path to node n; draft row n is the
 *     draft's logits there, from which node n's children were drawn
 *     independently (with replacement).
 *   - the walk starts at the root.  At node c with children x_1..x_m (in
 *     node-index order), child i is one ordinary accept test against the
 *     current distribution p_i of the target, with the draft q = q_c:
 *     accept with probability min(1, p_i(x_i) / q(x_i)); p_1 = p_c and after
 *     a rejection p_{i+1} = norm(max(0, p_i - q)) (the correction of the
 *     first page's step "Stop at the first rejection", applied to the next
 *     sibling instead of ending the round).  Written with running constants:
 *     p_i = max(0, p - C_i q) / M_i, C_1 = 0, M_1 = 1,
 *     C_{i+1} = C_i + M_i, M_{i+1} = sum_x max(0, p - C_{i+1} q).
 *   - an accepted child becomes the current node (its token is emitted);
 *     when every child is rejected, or c is a leaf, one token is drawn from
 *     the current distribution p_{m+1} (for a leaf: p_c, the bonus token) and
 *     the walk ends.  Every sibling test is one speculative-sampling step of
 *     target p_i against draft q, whose output law is p_i, so by induction
 *     the emitted token at each node follows p_c.
 *   - a tree in which every node has at most one child is the chain: the
 *     walk then equals spec_verify_ref_mt step for step.
 *   - T == 0: at node c the child (lowest index) whose token is the target's
 *     argmax is accepted; if none, the argmax is emitted and the walk ends.
 *   - rows are read (and checked) only as the walk visits them: target row c
 *     at every visited node, draft row c at a visited node with children when
 *     T > 0.  Sequence errors: T invalid (as spec_verify_ref_mt); n_nodes
 *     outside [1, N]; for 1 <= n < n_nodes, parent[n] outside [0, n) or
 *     tokens[n] outside [0, V); a visited row that holds NaN or +inf or is
 *     all -inf; q(x_i) <= 0 for a tested child.
 *   - M_{i+1} <= 0 after a rejection (impossible in exact arithmetic, where
 *     M_{i+1} >= M_2 (1 - q(S)) > 0 with S = {x : p(x) > q(x)}) ends the
 *     sibling tests and the draw falls back to p_c, like the chain's
 *     rounding fallback.
 */
typedef struct {
    const void *target;       /* [B, N, V] */
    const void *draft;        /* [B, N, V] */
    int dtype;
    const int32_t *parent;    /* [B, N] */
    const int32_t *tokens;    /* [B, N] */
    const int32_t *n_nodes;   /* [B] */
    const double *u_accept;   /* [B, N] */
    const double *u_resample; /* [B] */
    const double *temperature;/* [B] */
    int64_t N, V;
    int32_t *out_tokens;      /* [B, N] */
    int32_t *out_nodes;       /* [B, N] */
    int32_t *out_num_accepted;/* [B] */
    double *trace;            /* [B, N+3] or NULL */
    int64_t b0, b1;
    int status;
} ref_tree_job_t;

/* max(0, p - C q) into w; returns the total.  C == 0 copies p. */
static double ref_tree_residual(const double *p, const double *q, double C, int64_t V,
                                double *w)
{
    double M = 0.0;
    for (int64_t x = 0; x < V; ++x) {
        double d = (C == 0.0) ? p[x] : p[x] - C * q[x];
        w[x] = d > 0.0 ? d : 0.0;
        M += w[x];
    }
    return M;
}

/* Returns 0 on success, 1 if the sequence is an error row. */
static int ref_tree_sequence(ref_tree_job_t *J, int64_t b, double *t, double *d, double *p,
                             double *q, double *w)
{
    const int64_t N = J->N, V = J->V;
    const double T = J->temperature[b];
    const int32_t *par = J->parent + b * N, *tok = J->tokens + b * N;
    int32_t *ot = J->out_tokens + b * N, *on = J->out_nodes + b * N;
    double *tr = J->trace ? J->trace + b * (N + 3) : NULL;
    if (tr)
        for (int64_t i = 0; i < N + 3; ++i)
            tr[i] = NAN;

    if (isnan(T) || T < 0 || isinf(T) || (T > 0 && T < (double)FLT_MIN))
        return 1;
    const int64_t n = J->n_nodes[b];
    if (n < 1 || n > N)
        return 1;
    for (int64_t i = 1; i < n; ++i) {
        if (par[i] < 0 || par[i] >= i)
            return 1;
        if (tok[i] < 0 || tok[i] >= V)
            return 1;
    }

    int64_t c = 0, depth = 0, token = -1;
    for (;;) {
        ref_load_row(J->target, J->dtype, (size_t)(b * N + c), V, t);
        if (ref_row_invalid(t, V))
            return 1;
        int64_t first_child = -1;
        for (int64_t i = c + 1; i < n; ++i)
            if (par[i] == c) {
                first_child = i;
                break;
            }
        int64_t next = -1;
        if (T == 0) {
            int64_t a;
            ref_max_argmax(t, V, &a);
            for (int64_t i = c + 1; i < n; ++i)
                if (par[i] == c && tok[i] == a) {
                    next = i;
                    break;
                }
            if (next < 0) {
                token = a;
                break;
            }
        } else {
            spec_ref_softmax(t, V, T, p);
            double C = 0.0, M = 1.0;
            if (first_child >= 0) {
                ref_load_row(J->draft, J->dtype, (size_t)(b * N + c), V, d);
                if (ref_row_invalid(d, V))
                    return 1;
                spec_ref_softmax(d, V, T, q);
                for (int64_t i = first_child; i < n; ++i) {
                    if (par[i] != c)
                        continue;
                    const double Q = q[tok[i]];
                    if (Q <= 0.0)
                        return 1;
                    double num = p[tok[i]] - C * Q;
                    if (num < 0.0)
                        num = 0.0;
                    const double ratio = num / (M * Q);
                    if (tr)
                        tr[i] = ratio < 1.0 ? ratio : 1.0;
                    if (ratio >= 1.0 || J->u_accept[b * N + i] < ratio) {
                        next = i;
                        break;
                    }
                    C += M;
                    M = ref_tree_residual(p, q, C, V, w);
                    if (!(M > 0.0)) {
                        C = 0.0; /* rounding-only fallback: draw from p_c */
                        break;
                    }
                }
            }
            if (next < 0) {
                double R = ref_tree_residual(p, q, C, V, w);
                if (!(R > 0.0))
                    memcpy(w, p, (size_t)V * sizeof(double));
                double cell[3];
                token = spec_ref_inverse_cdf(w, V, J->u_resample[b], cell);
                if (token < 0)
                    return 1;
                if (tr) {
                    tr[N] = cell[0];
                    tr[N + 1] = cell[1];
                    tr[N + 2] = cell[2];
                }
                break;
            }
        }
        on[depth] = (int32_t)next;
        ot[depth] = tok[next];
        ++depth;
        c = next;
    }
    ot[depth] = (int32_t)token;
    for (int64_t i = depth + 1; i < N; ++i)
        ot[i] = -1;
    for (int64_t i = depth; i < N; ++i)
        on[i] = -1;
    J->out_num_accepted[b] = (int32_t)depth;
    return 0;
}

static void *ref_tree_worker(void *arg)
{
    ref_tree_job_t *J = (ref_tree_job_t *)arg;
    size_t n = (size_t)J->V;
    double *buf = (double *)malloc(5 * n * sizeof(double));
    if (!buf) {
        J->status = REF_ENOMEM;
        return NULL;
    }
    double *t = buf, *d = buf + n, *p = buf + 2 * n, *q = buf + 3 * n, *w = buf + 4 * n;
    for (int64_t b = J->b0; b < J->b1; ++b) {
        if (ref_tree_sequence(J, b, t, d, p, q, w)) {
            for (int64_t i = 0; i < J->N; ++i) {
                J->out_tokens[b * J->N + i] = -1;
                J->out_nodes[b * J->N + i] = -1;
            }
            J->out_num_accepted[b] = -1;
        }
    }
    free(buf);
    J->status = REF_OK;
    return NULL;
}

/*
 * Tree verification of B sequences of up to N nodes each (see above), split
 * over `nthreads` host threads.  target and draft are [B, N, V] (fp32 or bf16
 * bit patterns); parent, tokens [B, N] int32 (entry 0 unused); n_nodes [B];
 * u_accept [B, N] (entry n drives node n's test); u_resample [B]; T [B].
 * Outputs: out_tokens [B, N] (the accepted path's tokens, the drawn token,
 * then -1), out_nodes [B, N] (the accepted path's node indices, then -1),
 * out_num_accepted [B] (path length; -1 on a sequence error).  trace
 * (nullable) [B, N+3]: min(1, ratio) of each tested node (NaN elsewhere),
 * then the draw's cell [lo, hi) in u-units and its total (NaN for greedy).
 */
int spec_verify_tree_ref_mt(const void *target, const void *draft, int dtype,
                            const int32_t *parent, const int32_t *tokens,
                            const int32_t *n_nodes, const double *u_accept,
                            const double *u_resample, const double *temperature,
                            int64_t B, int64_t N, int64_t V,
                            int32_t *out_tokens, int32_t *out_nodes,
                            int32_t *out_num_accepted, double *trace, int nthreads)
{
    if (!target || !draft || !parent || !tokens || !n_nodes || !u_accept || !u_resample ||
        !temperature || !out_tokens || !out_nodes || !out_num_accepted)
        return REF_EINVAL;
    if (B < 0 || N < 1 || V < 2 || (dtype != REF_F32 && dtype != REF_BF16))
        return REF_EINVAL;
    if (B == 0)
        return REF_OK;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > B)
        nthreads = (int)B;
    ref_tree_job_t *jobs = (ref_tree_job_t *)calloc((size_t)nthreads, sizeof *jobs);
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return REF_ENOMEM;
    }
    for (int w = 0; w < nthreads; ++w) {
        ref_tree_job_t *J = &jobs[w];
        J->target = target;
        J->draft = draft;
        J->dtype = dtype;
        J->parent = parent;
        J->tokens = tokens;
        J->n_nodes = n_nodes;
        J->u_accept = u_accept;
        J->u_resample = u_resample;
        J->temperature = temperature;
        J->N = N;
        J->V = V;
        J->out_tokens = out_tokens;
        J->out_nodes = out_nodes;
        J->out_num_accepted = out_num_accepted;
        J->trace = trace;
        J->b0 = B * w / nthreads;
        J->b1 = B * (w + 1) / nthreads;
    }
    int started = 0;
    if (nthreads > 1)
        for (int w = 0; w < nthreads; ++w) {
            if (pthread_create(&th[w], NULL, ref_tree_worker, &jobs[w]) != 0)
                break;
            ++started;
        }
    for (int w = 0; w < started; ++w)
        pthread_join(th[w], NULL);
    for (int w = started; w < nthreads; ++w)
        ref_tree_worker(&jobs[w]);
    int status = REF_OK;
    for (int w = 0; w < nthreads; ++w)
        if (jobs[w].status != REF_OK)
            status = jobs[w].status;
    free(jobs);
    free(th);
    return status;
}
