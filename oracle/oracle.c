/*
 * oracle.c -- plain, slow, float64 CPU oracle for the batched verify-and-sample
 * step of speculative decoding and for the cache side of Saguaro (speculative
 * speculative decoding).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library; neither includes the other.
 *
 * Every quantity is computed in double with plain sequential loops in token-id
 * order.  Stored logits (fp32 or bf16 bit patterns) are widened exactly to
 * double before any arithmetic.  Each function cites the passage it follows:
 *   [SD]   "Speculative decoding" (brentwoodlivery.com), sections "The Algorithm
 *          (Step-by-Step)", "Derivation of Acceptance Criterion", "Temperature and
 *          Sampling", "Batching Speculation".
 *   [WHY]  "Why does speculative decoding exist?" (til.phipham141.dev), section
 *          "How it works", Fix 2 / Fix 3 (bonus token, greedy rule).
 *   [SSD]  "Speculative Speculative Decoding" notes (papernotes.org), section
 *          "关键设计" items 1 (fan-out), 2 (SAGUARO sampling) and 3 (batch-aware
 *          fallback, random-token backup), and the SSD
 *          iteration of section "整体框架" (outcome (k, t*), cache S_T, hit test).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - accept test: accept x~ iff u * q(x~) < p(x~) with u in [0,1)  (equivalent to
 *     u < min(1, p/q) without a division);
 *   - the bonus draw uses u[K] whatever the accepted length is;
 *   - the residual / p CDF runs over ascending token id and picks the first token
 *     whose cumulative weight exceeds u * Z (strictly);
 *   - Z == 0 in the residual: the bonus is drawn from p at that row instead;
 *   - greedy (tau == 0): compare raw stored logits, lowest id wins ties;
 *   - fan-out: real-valued F_k rounded by the largest-remainder method;
 *   - uniform fan-out: floor(budget/(K+1)) each, remainder to the lowest k;
 *   - random backup token: floor(u * V) for a supplied uniform u in [0, 1);
 *   - cache scores: (p_k - q_k)^+ for k < K, p_K for k = K (tau > 0); raw target
 *     logits with the drafted token excluded (tau == 0);
 *   - draft-only cache keys: raw draft logits of row k (of K+1 draft rows), the
 *     drafted token left out for k < K; the reshape at position k uses F = F_k.
 * Where the pages are silent (which uniform draws the bonus, the CDF order and
 * boundary, the Z == 0 fallback) they fix only the law of the draw: the tests pin
 * that law (chi-square, exact enumeration) and pin the chosen readings token by
 * token against numpy's inverse CDF of scipy's softmax on the same uniforms; the
 * Z == 0 fallback also against its hit probability, the cached mass of p_a.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1

/* --------------------------------------------------------------------------
 * Storage decoding: one stored logit widened exactly to double.
 * ------------------------------------------------------------------------ */
static double stored_value(const void *base, int dtype, int64_t idx)
{
    if (dtype == OR_F32)
        return (double)((const float *)base)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static void load_row(const void *base, int dtype, int64_t row_start, int V, double *z)
{
    for (int t = 0; t < V; ++t)
        z[t] = stored_value(base, dtype, row_start + t);
}

/* --------------------------------------------------------------------------
 * [SD] "Temperature and Sampling": p_tau = softmax(logits / tau).
 *   p(t) = exp(z_t/tau - m) / sum_j exp(z_j/tau - m),  m = max_j z_j/tau.
 * The shift m cancels; it only keeps exp() in range.
 * ------------------------------------------------------------------------ */
void oracle_softmax(const double *z, int V, double tau, double *p)
{
    double m = -INFINITY;
    for (int t = 0; t < V; ++t)
        if (z[t] / tau > m)
            m = z[t] / tau;
    double S = 0.0;
    for (int t = 0; t < V; ++t) {
        p[t] = exp(z[t] / tau - m);
        S += p[t];
    }
    for (int t = 0; t < V; ++t)
        p[t] /= S;
}

/* --------------------------------------------------------------------------
 * Ranking helper: order tokens by (score descending, token id ascending); an
 * excluded token ranks below every other token.  qsort is the library sort.
 * ------------------------------------------------------------------------ */
typedef struct {
    double score;
    int id;
    int excluded;
} ranked_t;

static int rank_cmp(const void *pa, const void *pb)
{
    const ranked_t *a = (const ranked_t *)pa, *b = (const ranked_t *)pb;
    if (a->excluded != b->excluded)
        return a->excluded ? 1 : -1;
    if (a->score > b->score)
        return -1;
    if (a->score < b->score)
        return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id);
}

/* Fills order[0..V) with token ids sorted by (score desc, id asc), excluded last.
 * excl_id < 0: nothing excluded. */
static void rank_tokens(const double *score, int V, int excl_id, ranked_t *work, int *order)
{
    for (int t = 0; t < V; ++t) {
        work[t].score = score[t];
        work[t].id = t;
        work[t].excluded = (t == excl_id);
    }
    qsort(work, (size_t)V, sizeof(ranked_t), rank_cmp);
    for (int t = 0; t < V; ++t)
        order[t] = work[t].id;
}

/* top-F of raw logits, ties to the lowest id: ids written to out[0..F). */
void oracle_topf(const double *z, int V, int F, int *out)
{
    ranked_t *work = (ranked_t *)malloc(sizeof(ranked_t) * (size_t)V);
    int *order = (int *)malloc(sizeof(int) * (size_t)V);
    rank_tokens(z, V, -1, work, order);
    for (int i = 0; i < F && i < V; ++i)
        out[i] = order[i];
    free(order);
    free(work);
}

/* --------------------------------------------------------------------------
 * [SSD] item 2, SAGUARO sampling: sigma_{F,C}(z)_t is proportional to
 * C*exp(z_t) when t is among the F largest draft logits, exp(z_t) otherwise.
 * Temperature is applied first (z -> z/tau); the top-F set is taken on the raw
 * logits, which gives the same set for every tau > 0.
 *   q'(t) = c_t exp(z_t/tau - m) / sum_j c_j exp(z_j/tau - m),  c_t in {C, 1}.
 * m is the largest z_j/tau over tokens with c_j > 0 (any shift cancels).
 * Returns 0, or -1 when every token has weight zero (C == 0 and F >= V).
 * member_out (optional): 1 for the top-F tokens.
 * ------------------------------------------------------------------------ */
int oracle_sigma(const double *z, int V, double tau, int F, double C, double *q,
                 unsigned char *member_out)
{
    unsigned char *member = (unsigned char *)calloc((size_t)V, 1);
    if (F > 0) {
        int Fe = F < V ? F : V;
        int *ids = (int *)malloc(sizeof(int) * (size_t)Fe);
        oracle_topf(z, V, Fe, ids);
        for (int i = 0; i < Fe; ++i)
            member[ids[i]] = 1;
        free(ids);
    }
    double m = -INFINITY;
    for (int t = 0; t < V; ++t) {
        double c = member[t] ? C : 1.0;
        if (c > 0.0 && z[t] / tau > m)
            m = z[t] / tau;
    }
    if (m == -INFINITY) {
        free(member);
        return -1;
    }
    double S = 0.0;
    for (int t = 0; t < V; ++t) {
        double c = member[t] ? C : 1.0;
        q[t] = c * exp(z[t] / tau - m);
        S += q[t];
    }
    for (int t = 0; t < V; ++t)
        q[t] /= S;
    if (member_out)
        memcpy(member_out, member, (size_t)V);
    free(member);
    return 0;
}

/* --------------------------------------------------------------------------
 * [SSD] item 1, geometric fan-out.  For k < K: F_k = F_0 * a_p^{k/(1+r)};
 * F_K = F_0 * a_p^{K/(1+r)} * (1-a_p)^{-1/(1+r)}; sum_k F_k <= budget.
 * F_0 is the largest value that fits the budget (sum = budget before
 * rounding); the real values x_k are made integers by the largest-remainder
 * method (floor, then +1 to the largest fractional parts, lowest k on ties),
 * so sum F_k == budget; finally each F_k is clamped to V.
 * Writes F[0..K], off[0..K+1] (exclusive prefix sums).  Returns 0 or -1.
 * x_out (optional): the real-valued x_k before rounding.
 * ------------------------------------------------------------------------ */
int oracle_fanout(int K, int budget, double a_p, double r, int V, int *F, int *off,
                  double *x_out)
{
    if (K < 1 || budget < 0 || !(a_p > 0.0 && a_p < 1.0) || !(r > -1.0) || V < 1)
        return -1;
    double *w = (double *)malloc(sizeof(double) * (size_t)(K + 1));
    double *x = (double *)malloc(sizeof(double) * (size_t)(K + 1));
    double wsum = 0.0;
    for (int k = 0; k < K; ++k) {
        w[k] = pow(a_p, (double)k / (1.0 + r));
        wsum += w[k];
    }
    w[K] = pow(a_p, (double)K / (1.0 + r)) * pow(1.0 - a_p, -1.0 / (1.0 + r));
    wsum += w[K];
    double F0 = (double)budget / wsum;
    long assigned = 0;
    for (int k = 0; k <= K; ++k) {
        x[k] = F0 * w[k];
        F[k] = (int)floor(x[k]);
        assigned += F[k];
    }
    long left = (long)budget - assigned;
    unsigned char *bumped = (unsigned char *)calloc((size_t)(K + 1), 1);
    while (left > 0) {
        int best = -1;
        double best_frac = -1.0;
        for (int k = 0; k <= K; ++k) {
            double frac = x[k] - floor(x[k]);
            if (!bumped[k] && frac > best_frac) {
                best_frac = frac;
                best = k;
            }
        }
        if (best < 0) { /* every entry bumped once: cannot happen (left <= K) */
            memset(bumped, 0, (size_t)(K + 1));
            continue;
        }
        F[best] += 1;
        bumped[best] = 1;
        --left;
    }
    off[0] = 0;
    for (int k = 0; k <= K; ++k) {
        if (F[k] > V)
            F[k] = V;
        off[k + 1] = off[k] + F[k];
    }
    if (x_out)
        memcpy(x_out, x, sizeof(double) * (size_t)(K + 1));
    free(bumped);
    free(x);
    free(w);
    return 0;
}

/* ------------------------------------------------------------------------
 * [SSD] item 1, uniform fan-out: the allocation the geometric shape is
 * compared with (and beats at higher temperature): the budget is spread evenly
 * over the K+1 accepted lengths.  Reading: equal integer shares floor(budget/(K+1)),
 * the remainder one slot each to the lowest k, each share clamped to V.
 * Writes F[0..K], off[0..K+1].  Returns 0 or -1.
 * ------------------------------------------------------------------------ */
int oracle_fanout_uniform(int K, int budget, int V, int *F, int *off)
{
    if (K < 1 || budget < 0 || V < 1)
        return -1;
    off[0] = 0;
    for (int k = 0; k <= K; ++k) {
        int f = budget / (K + 1);
        if (k < budget % (K + 1))
            f += 1;
        if (f > V)
            f = V;
        F[k] = f;
        off[k + 1] = off[k] + f;
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * [SSD] item 3, fast backup speculator: at large batch the sequences that miss
 * the cache are re-drafted by a very fast, low-quality speculator; the notes
 * name random tokens as the one implemented.  Reading: token i of sequence b
 * is floor(u[b, i] * V) (clamped to V-1) for a uniform u in [0, 1) supplied by
 * the caller, for every sequence with hit[b] == 0; other rows are untouched.
 * ------------------------------------------------------------------------ */
void oracle_backup_fill(const unsigned char *hit, const float *u, int B, int K, int V, int *next)
{
    for (int b = 0; b < B; ++b) {
        if (hit[b])
            continue;
        for (int i = 0; i < K; ++i) {
            double x = (double)u[(size_t)b * K + i] * (double)V;
            long t = (long)floor(x);
            if (t > V - 1)
                t = V - 1;
            if (t < 0)
                t = 0;
            next[(size_t)b * K + i] = (int)t;
        }
    }
}

/* --------------------------------------------------------------------------
 * Per-sequence scratch.
 * ------------------------------------------------------------------------ */
typedef struct {
    int V;
    double *zt, *zd;    /* one target row, one draft row (raw logits) */
    double *p, *q;      /* their (reshaped) temperature softmaxes */
    double *w;          /* residual / bonus weights */
    double *score;
    ranked_t *work;
    int *order;
} scratch_t;

static int scratch_init(scratch_t *s, int V)
{
    s->V = V;
    s->zt = (double *)malloc(sizeof(double) * (size_t)V);
    s->zd = (double *)malloc(sizeof(double) * (size_t)V);
    s->p = (double *)malloc(sizeof(double) * (size_t)V);
    s->q = (double *)malloc(sizeof(double) * (size_t)V);
    s->w = (double *)malloc(sizeof(double) * (size_t)V);
    s->score = (double *)malloc(sizeof(double) * (size_t)V);
    s->work = (ranked_t *)malloc(sizeof(ranked_t) * (size_t)V);
    s->order = (int *)malloc(sizeof(int) * (size_t)V);
    return (s->zt && s->zd && s->p && s->q && s->w && s->score && s->work && s->order) ? 0 : -1;
}

static void scratch_free(scratch_t *s)
{
    free(s->zt); free(s->zd); free(s->p); free(s->q);
    free(s->w); free(s->score); free(s->work); free(s->order);
}

/* Problem description shared by every batched entry point. */
typedef struct {
    int B, K, V, dtype;
    const void *tgt;            /* [B, K+1, V] stored logits */
    const void *drf;            /* [B, drf_rows, V] stored logits */
    int drf_rows;               /* rows per sequence in drf (K or K+1) */
    const int *tokens;          /* [B, K] drafted tokens x~ */
    const float *uniforms;      /* [B, K+1] */
    const float *tau;           /* [B] temperatures */
    int reshape_F;              /* sigma_{F,C} on the draft rows (0 = none) */
    const int *reshape_Fk;      /* [K] per-position F (overrides reshape_F), or NULL */
    double reshape_C;
} problem_t;

/* p = softmax(target row i / tau); q = (reshaped) softmax(draft row i / tau). */
static void target_probs(const problem_t *P, int b, int i, double tau, scratch_t *s)
{
    load_row(P->tgt, P->dtype, ((int64_t)b * (P->K + 1) + i) * P->V, P->V, s->zt);
    oracle_softmax(s->zt, P->V, tau, s->p);
}

static int draft_probs(const problem_t *P, int b, int i, double tau, scratch_t *s)
{
    load_row(P->drf, P->dtype, ((int64_t)b * P->drf_rows + i) * P->V, P->V, s->zd);
    const int F = P->reshape_Fk ? P->reshape_Fk[i] : P->reshape_F;
    if (F > 0)
        return oracle_sigma(s->zd, P->V, tau, F, P->reshape_C, s->q, NULL);
    oracle_softmax(s->zd, P->V, tau, s->q);
    return 0;
}

/* Greedy target decision of row i: argmax of the raw stored logits, lowest id
 * on ties ([WHY] Fix 2: greedy acceptance is "draft token == target argmax"). */
static int row_argmax(const double *z, int V)
{
    int best = 0;
    for (int t = 1; t < V; ++t)
        if (z[t] > z[best])
            best = t;
    return best;
}

/* Inverse CDF over ascending token id: the first t whose cumulative weight
 * exceeds T = u * Z.  Returns t and the margin (distance from T to the nearer
 * edge of t's CDF interval, divided by Z). */
static int cdf_invert(const double *w, int V, double u, double *margin)
{
    double Z = 0.0;
    for (int t = 0; t < V; ++t)
        Z += w[t];
    double T = u * Z;
    double below = 0.0, cum = 0.0;
    int pick = -1, last_pos = -1;
    for (int t = 0; t < V; ++t) {
        if (w[t] > 0.0)
            last_pos = t;
        below = cum;
        cum += w[t];
        if (cum > T) {
            pick = t;
            break;
        }
    }
    if (pick < 0) { /* T reached the total only through rounding: last positive */
        pick = last_pos;
        *margin = 0.0;
        return pick;
    }
    double m1 = T - below, m2 = cum - T;
    *margin = (m1 < m2 ? m1 : m2) / Z;
    return pick;
}

/* Outputs of one verification. */
typedef struct {
    int a, bonus;
    double *p_tok, *q_tok;      /* [K] */
    double *acc_margin;         /* [K] */
    double bonus_margin;
    double Z;                   /* residual mass at row a (1 when a == K) */
} verify_out_t;

/* --------------------------------------------------------------------------
 * [SD] "The Algorithm (Step-by-Step)", step 3, one sequence:
 *   for each drafted token in order, accept with probability min(1, p/q);
 *   on the first rejection at i, draw the bonus from max(0, p_i - q_i)/Z and
 *   discard the rest; if all K are accepted, draw the bonus from p at row K.
 * [SD] "Temperature and Sampling": p and q are the temperature softmaxes.
 * [WHY] Fix 2: tau == 0 accepts iff the drafted token is the target argmax,
 * and the bonus is the target argmax at the stopping row.
 * Returns 0, or -1 on an invalid sequence (bad token id or temperature).
 * ------------------------------------------------------------------------ */
static int verify_sequence(const problem_t *P, int b, scratch_t *s, verify_out_t *o)
{
    const int K = P->K, V = P->V;
    const double tau = (double)P->tau[b];
    const int *x = P->tokens + (int64_t)b * K;
    const float *u = P->uniforms + (int64_t)b * (K + 1);
    for (int i = 0; i < K; ++i) {
        o->p_tok[i] = NAN;
        o->q_tok[i] = NAN;
        o->acc_margin[i] = INFINITY;
    }
    o->a = -1;
    o->bonus = -1;
    o->bonus_margin = INFINITY;
    o->Z = NAN;
    if (!(tau >= 0.0))
        return -1;
    for (int i = 0; i < K; ++i)
        if (x[i] < 0 || x[i] >= V)
            return -1;

    if (tau == 0.0) {
        int a = K;
        for (int i = 0; i < K; ++i) {
            load_row(P->tgt, P->dtype, ((int64_t)b * (K + 1) + i) * V, V, s->zt);
            int am = row_argmax(s->zt, V);
            o->p_tok[i] = (am == x[i]) ? 1.0 : 0.0;
            o->q_tok[i] = 1.0;
            if (am != x[i]) {
                a = i;
                o->bonus = am;
                break;
            }
        }
        if (a == K) {
            load_row(P->tgt, P->dtype, ((int64_t)b * (K + 1) + K) * V, V, s->zt);
            o->bonus = row_argmax(s->zt, V);
        }
        o->a = a;
        o->Z = 1.0;
        return 0;
    }

    int a = K;
    for (int i = 0; i < K; ++i) {
        target_probs(P, b, i, tau, s);
        if (draft_probs(P, b, i, tau, s) != 0)
            return -1;
        double pt = s->p[x[i]], qt = s->q[x[i]];
        o->p_tok[i] = pt;
        o->q_tok[i] = qt;
        double ui = (double)u[i];
        int accept = (ui * qt < pt);
        o->acc_margin[i] = (pt >= qt) ? INFINITY : fabs(ui - pt / qt);
        if (!accept) {
            a = i;
            break;
        }
    }
    /* s->p and s->q hold row a when a < K. */
    if (a < K) {
        double Z = 0.0;
        for (int t = 0; t < V; ++t) {
            double d = s->p[t] - s->q[t];
            s->w[t] = d > 0.0 ? d : 0.0;
            Z += s->w[t];
        }
        if (Z == 0.0) { /* p == q everywhere at this row: draw from p */
            memcpy(s->w, s->p, sizeof(double) * (size_t)V);
            Z = 1.0;
        }
        o->Z = Z;
    } else {
        target_probs(P, b, K, tau, s);
        memcpy(s->w, s->p, sizeof(double) * (size_t)V);
        o->Z = 1.0;
    }
    o->bonus = cdf_invert(s->w, V, (double)u[K], &o->bonus_margin);
    o->a = a;
    return 0;
}

/* --------------------------------------------------------------------------
 * [SSD] item 1 + item 2 text: per accepted length k the cache holds the F_k
 * bonus tokens most likely to be drawn at that outcome.  tau > 0: k < K ranks
 * the residual (p_k - q_k)^+, k == K ranks p_K.  tau == 0: the bonus is the
 * target argmax, so rank the raw target logits of row k, excluding the
 * drafted token x~_k for k < K (a rejection at k means argmax != x~_k).
 * Writes cache_tok[off[k] .. off[k+1]) in rank order, the score of each entry,
 * and the margin (gap between the last kept and first dropped score; +inf
 * when exact).
 * ------------------------------------------------------------------------ */
static int cache_sequence(const problem_t *P, int b, const int *off, scratch_t *s,
                          int *cache_tok, double *cache_score, double *cache_margin)
{
    const int K = P->K, V = P->V;
    const double tau = (double)P->tau[b];
    const int *x = P->tokens + (int64_t)b * K;
    if (!(tau >= 0.0))
        return -1;
    for (int i = 0; i < K; ++i)
        if (x[i] < 0 || x[i] >= V)
            return -1;
    for (int k = 0; k <= K; ++k) {
        int Fk = off[k + 1] - off[k];
        int excl = -1;
        if (tau == 0.0) {
            load_row(P->tgt, P->dtype, ((int64_t)b * (K + 1) + k) * V, V, s->zt);
            memcpy(s->score, s->zt, sizeof(double) * (size_t)V);
            if (k < K)
                excl = x[k];
        } else if (k < K) {
            target_probs(P, b, k, tau, s);
            if (draft_probs(P, b, k, tau, s) != 0)
                return -1;
            for (int t = 0; t < V; ++t) {
                double d = s->p[t] - s->q[t];
                s->score[t] = d > 0.0 ? d : 0.0;
            }
        } else {
            target_probs(P, b, K, tau, s);
            memcpy(s->score, s->p, sizeof(double) * (size_t)V);
        }
        rank_tokens(s->score, V, excl, s->work, s->order);
        for (int j = 0; j < Fk && j < V; ++j) {
            cache_tok[off[k] + j] = s->order[j];
            cache_score[off[k] + j] = (s->order[j] == excl) ? -INFINITY : s->score[s->order[j]];
        }
        double margin = INFINITY;
        if (tau > 0.0 && Fk > 0 && Fk < V) {
            double lo = s->score[s->order[Fk - 1]], hi = s->score[s->order[Fk]];
            if (s->order[Fk] != excl && lo != hi)
                margin = lo - hi;
        }
        cache_margin[k] = margin;
    }
    return 0;
}

/* [SSD] "整体框架": the outcome v = (k, t*) hits iff it is in S_T, i.e. t* is in
 * the cached segment of accepted length k.  slot = position in the row, else -1. */
static void lookup_sequence(const int *cache_row, const int *off, int a, int bonus,
                            unsigned char *hit, int *slot)
{
    *hit = 0;
    *slot = -1;
    if (a < 0)
        return;
    for (int j = off[a]; j < off[a + 1]; ++j) {
        if (cache_row[j] == bonus) {
            *hit = 1;
            *slot = j;
            return;
        }
    }
}

/* --------------------------------------------------------------------------
 * Batched entry points (ctypes).  Each processes sequences [b0, b1) so that a
 * caller may split a batch across host threads.
 * ------------------------------------------------------------------------ */
static problem_t make_problem(int B, int K, int V, int dtype, const void *tgt, const void *drf,
                              int drf_rows, const int *tokens, const float *uniforms,
                              const float *tau, int reshape_F, const int *reshape_Fk,
                              double reshape_C)
{
    problem_t P;
    P.B = B; P.K = K; P.V = V; P.dtype = dtype;
    P.tgt = tgt; P.drf = drf; P.drf_rows = drf_rows;
    P.tokens = tokens; P.uniforms = uniforms; P.tau = tau;
    P.reshape_F = reshape_F; P.reshape_Fk = reshape_Fk; P.reshape_C = reshape_C;
    return P;
}

/* [SD] step 3 over a batch ([SD] "Batching Speculation": every sequence is
 * verified independently; shorter outcomes are simply shorter).
 * Outputs per sequence: accept_len, bonus, p_tok/q_tok [K] (NaN past a),
 * acc_margin [K], bonus_margin, Z.  Returns the number of invalid sequences. */
int oracle_verify(int b0, int b1, int B, int K, int V, int dtype, const void *tgt,
                  const void *drf, int drf_rows, const int *tokens, const float *uniforms,
                  const float *tau, int reshape_F, const int *reshape_Fk, double reshape_C,
                  int *accept_len, int *bonus, double *p_tok, double *q_tok,
                  double *acc_margin, double *bonus_margin, double *Z)
{
    problem_t P = make_problem(B, K, V, dtype, tgt, drf, drf_rows, tokens, uniforms, tau,
                               reshape_F, reshape_Fk, reshape_C);
    scratch_t s;
    if (scratch_init(&s, V) != 0) {
        scratch_free(&s);
        return -1;
    }
    int bad = 0;
    for (int b = b0; b < b1; ++b) {
        verify_out_t o;
        o.p_tok = p_tok + (int64_t)b * K;
        o.q_tok = q_tok + (int64_t)b * K;
        o.acc_margin = acc_margin + (int64_t)b * K;
        if (verify_sequence(&P, b, &s, &o) != 0)
            ++bad;
        accept_len[b] = o.a;
        bonus[b] = o.bonus;
        bonus_margin[b] = o.bonus_margin;
        Z[b] = o.Z;
    }
    scratch_free(&s);
    return bad;
}

/* Cache build over a batch: cache_tok [B, budget], cache_score [B, budget],
 * cache_margin [B, K+1].  off [K+2] from the fan-out. */
int oracle_build_cache(int b0, int b1, int B, int K, int V, int dtype, const void *tgt,
                       const void *drf, int drf_rows, const int *tokens, const float *tau,
                       int reshape_F, const int *reshape_Fk, double reshape_C, const int *off,
                       int budget, int *cache_tok, double *cache_score, double *cache_margin)
{
    problem_t P = make_problem(B, K, V, dtype, tgt, drf, drf_rows, tokens, NULL, tau,
                               reshape_F, reshape_Fk, reshape_C);
    scratch_t s;
    if (scratch_init(&s, V) != 0) {
        scratch_free(&s);
        return -1;
    }
    int bad = 0;
    for (int b = b0; b < b1; ++b) {
        int *row = cache_tok + (int64_t)b * budget;
        double *srow = cache_score + (int64_t)b * budget;
        for (int j = 0; j < budget; ++j) {
            row[j] = -1;
            srow[j] = NAN;
        }
        if (cache_sequence(&P, b, off, &s, row, srow, cache_margin + (int64_t)b * (K + 1)) != 0)
            ++bad;
    }
    scratch_free(&s);
    return bad;
}

/* Hit test over a batch. */
void oracle_lookup(int B, int budget, const int *off, const int *cache_tok,
                   const int *accept_len, const int *bonus, unsigned char *hit, int *slot)
{
    for (int b = 0; b < B; ++b)
        lookup_sequence(cache_tok + (int64_t)b * budget, off, accept_len[b], bonus[b], hit + b,
                        slot + b);
}

/* --------------------------------------------------------------------------
 * [SSD] item 2, cache keys chosen from the draft logits.  For sequence b and
 * accepted length k, segment k of the cache row holds the F_k tokens ranked
 * highest by raw draft logit (row k of drf [B, K+1, V]; ties to the lowest
 * id).  Reading: for k < K the drafted token x~_k is left out (after x~_k is
 * rejected the residual max(0, p - q) is zero there, so it is never the
 * bonus); a slot with no token left (F_k == V) holds -1.  tokens may be NULL.
 * ------------------------------------------------------------------------ */
int oracle_draft_cache(int B, int K, int V, int dtype, const void *drf, const int *tokens,
                       const int *off, int budget, int *cache_tok)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    ranked_t *work = (ranked_t *)malloc(sizeof(ranked_t) * (size_t)V);
    int *order = (int *)malloc(sizeof(int) * (size_t)V);
    if (!z || !work || !order) {
        free(z); free(work); free(order);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        for (int k = 0; k <= K; ++k) {
            load_row(drf, dtype, ((int64_t)b * (K + 1) + k) * V, V, z);
            int excl = (tokens && k < K) ? tokens[(int64_t)b * K + k] : -1;
            rank_tokens(z, V, excl, work, order);
            int *seg = cache_tok + (int64_t)b * budget + off[k];
            for (int j = 0; j < off[k + 1] - off[k]; ++j)
                seg[j] = (j < V && order[j] != excl) ? order[j] : -1;
        }
    }
    free(z); free(work); free(order);
    return 0;
}

/* --------------------------------------------------------------------------
 * Probability that the true outcome (a, t*) of one round is in the cache,
 * given the drafted tokens and the cache ([SSD] "整体框架": the round hits when
 * (a, t*) is among the cached outcomes; [SD] step 3 fixes the law of (a, t*)):
 *   tau > 0:  position i is accepted with probability min(1, p_i(x~_i) / q_i(x~_i));
 *             a rejection at k draws t* from max(0, p_k - q_k) / Z (from p_k
 *             when Z == 0), acceptance of all K draws t* from p_K; so
 *             P_hit = sum_k P(a = k) * (weight of segment k) / (total weight).
 *   tau == 0: a and t* are fixed by the target argmaxes; P_hit is 0 or 1.
 * q is sigma_{F,C} when reshape_F / reshape_Fk is given (as in oracle_verify).
 * Writes p_hit[b0..b1).  Returns the number of invalid sequences (-1 there).
 * ------------------------------------------------------------------------ */
int oracle_p_hit(int b0, int b1, int B, int K, int V, int dtype, const void *tgt,
                 const void *drf, int drf_rows, const int *tokens, const float *tau,
                 int reshape_F, const int *reshape_Fk, double reshape_C, const int *off,
                 int budget, const int *cache_tok, double *p_hit)
{
    problem_t P = make_problem(B, K, V, dtype, tgt, drf, drf_rows, tokens, NULL, tau,
                               reshape_F, reshape_Fk, reshape_C);
    scratch_t s;
    if (scratch_init(&s, V) != 0) {
        scratch_free(&s);
        return -1;
    }
    int bad = 0;
    for (int b = b0; b < b1; ++b) {
        const int *x = tokens + (int64_t)b * K;
        const int *row = cache_tok + (int64_t)b * budget;
        const double t = (double)tau[b];
        int ok = (t >= 0.0);
        for (int i = 0; i < K; ++i)
            if (x[i] < 0 || x[i] >= V)
                ok = 0;
        if (!ok) {
            p_hit[b] = -1.0;
            ++bad;
            continue;
        }
        if (t == 0.0) {
            int a = K, tstar = -1;
            for (int i = 0; i <= K; ++i) {
                load_row(tgt, dtype, ((int64_t)b * (K + 1) + i) * V, V, s.zt);
                int am = row_argmax(s.zt, V);
                if (i == K || am != x[i]) {
                    a = i;
                    tstar = am;
                    break;
                }
            }
            double h = 0.0;
            for (int j = off[a]; j < off[a + 1]; ++j)
                if (row[j] == tstar)
                    h = 1.0;
            p_hit[b] = h;
            continue;
        }
        double reach = 1.0, total = 0.0;
        for (int k = 0; k <= K && reach > 0.0; ++k) {
            double pa, acc = 1.0;
            target_probs(&P, b, k, t, &s);
            if (k < K) {
                if (draft_probs(&P, b, k, t, &s) != 0) {
                    ok = 0;
                    break;
                }
                double pt = s.p[x[k]], qt = s.q[x[k]];
                acc = (qt > 0.0) ? fmin(1.0, pt / qt) : (pt > 0.0 ? 1.0 : 0.0);
                pa = reach * (1.0 - acc);
                double Z = 0.0;
                for (int v = 0; v < V; ++v) {
                    s.w[v] = fmax(0.0, s.p[v] - s.q[v]);
                    Z += s.w[v];
                }
                if (Z == 0.0)
                    for (int v = 0; v < V; ++v)
                        s.w[v] = s.p[v];
            } else {
                pa = reach;
                for (int v = 0; v < V; ++v)
                    s.w[v] = s.p[v];
            }
            double W = 0.0, in = 0.0;
            for (int v = 0; v < V; ++v)
                W += s.w[v];
            for (int j = off[k]; j < off[k + 1]; ++j)
                if (row[j] >= 0 && row[j] < V)
                    in += s.w[row[j]];
            total += pa * (in / W);
            reach *= acc;
        }
        if (!ok) {
            p_hit[b] = -1.0;
            ++bad;
            continue;
        }
        p_hit[b] = total;
    }
    scratch_free(&s);
    return bad;
}

/* sigma_{F,C} over independent rows: q_out [rows, V] (may be NULL), member
 * flags [rows, V] (may be NULL). */
int oracle_reshape_rows(int r0, int r1, int V, int dtype, const void *logits, const float *tau,
                        int F, double C, double *q_out, unsigned char *member_out)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    unsigned char *mem = (unsigned char *)malloc((size_t)V);
    int bad = 0;
    for (int r = r0; r < r1; ++r) {
        load_row(logits, dtype, (int64_t)r * V, V, z);
        if (oracle_sigma(z, V, (double)tau[r], F, C, q, mem) != 0) {
            ++bad;
            continue;
        }
        if (q_out)
            memcpy(q_out + (int64_t)r * V, q, sizeof(double) * (size_t)V);
        if (member_out)
            memcpy(member_out + (int64_t)r * V, mem, (size_t)V);
    }
    free(mem);
    free(q);
    free(z);
    return bad;
}
