/*
 * Plain fp64 CPU oracle of the DFlash 2 path selector.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
 * baseline leg load this file's library. The product path never calls it and
 * shares no code with it: every quantity here is recomputed from its
 * definition, in double precision, with explicit loops, a full sort and no
 * blocking or fusion.
 *
 * Source of the method: the blog post "DFlash 2: Keep Drafting Parallel"
 * (Inco AI), section "A Lightweight Path Selector":
 *   - the drafter keeps its 16 best candidates at every draft position;
 *   - every adjacent pair (predecessor a, current candidate b) at position t
 *     gets the score  S_t(a,b) = U_t(b) + < A(a) (.) H(h_t), B(b) >,
 *     where U_t is the drafter's own logit, A and B give each token a
 *     256-wide embedding and H(h_t) is a gate computed from the position's
 *     hidden state;
 *   - a walk over the precomputed scores picks one path, starting from the
 *     last verified token;
 *   - the target model checks the block and keeps the accepted prefix.
 *
 * Readings taken where the pages are silent (listed with reasons in the
 * design notes):
 *   R1  A(a) = W_A E[a], B(b) = W_B E[b], H(h) = W_H h, with one shared token
 *       table E [V, d] and W_A, W_B, W_H of shape [e, d]; no bias, no norm.
 *   R2  U_t is the raw lm_head logit W[b] . h_t.
 *   R3  the walk is a max-sum (Viterbi) walk over the tables; the literal
 *       walk that takes the best successor at every step is kept as mode 1.
 *   R4  top-K order: value descending, then token id ascending.
 *   R5  Viterbi ties: the smallest predecessor rank wins; at the end the
 *       smallest final rank wins. Greedy ties: the smallest rank wins.
 *   R6  the only predecessor at the first draft position is the anchor x0.
 *   R8  accept length n = number of leading draft tokens equal to the
 *       target's argmax tokens; the emitted tokens are those n plus the
 *       target's token at position n (L+1 target columns).
 *
 * Indexing is 0-based: draft position t = 0 .. L-1 is the pages' position
 * t+1. All bf16 inputs arrive as raw bit patterns and are widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* U[n*V + v] = sum_i W[v, i] * H[n, i]: the lm_head logit of token v at
 * position n (the drafter's own logit, U_t(b) of the S_t equation). */
void oracle_logits(const uint16_t *W, const uint16_t *H, int64_t V, int64_t d, int64_t N,
                   double *U, int nthreads)
{
    double *h = (double *)malloc((size_t)(N * d) * sizeof(double));
    for (int64_t k = 0; k < N * d; ++k) h[k] = bf16_to_f64(H[k]);
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
    for (int64_t v = 0; v < V; ++v) {
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t i = 0; i < d; ++i) s += bf16_to_f64(W[v * d + i]) * h[n * d + i];
            U[n * V + v] = s;
        }
    }
    (void)nthreads;
    free(h);
}

typedef struct {
    double val;
    int32_t id;
} scored_token;

/* value descending, then id ascending (reading R4) */
static int cmp_scored(const void *pa, const void *pb)
{
    const scored_token *a = (const scored_token *)pa, *b = (const scored_token *)pb;
    if (a->val > b->val) return -1;
    if (a->val < b->val) return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id);
}

/* Keeps the K best tokens of one logit row by a full sort of all V entries.
 * margin = U_(K) - U_(K+1), the gap at the top-K boundary (+inf if K == V). */
void oracle_topk(const double *U, int64_t V, int K, int32_t *ids, double *vals, double *margin)
{
    scored_token *all = (scored_token *)malloc((size_t)V * sizeof(scored_token));
    for (int64_t v = 0; v < V; ++v) {
        all[v].val = U[v];
        all[v].id = (int32_t)v;
    }
    qsort(all, (size_t)V, sizeof(scored_token), cmp_scored);
    for (int k = 0; k < K; ++k) {
        ids[k] = all[k].id;
        vals[k] = all[k].val;
    }
    *margin = (K < V) ? all[K - 1].val - all[K].val : INFINITY;
    free(all);
}

/* out[r] = sum_i P[r, i] * x[i] for a bf16 matrix P [rows, d] and bf16 vector x:
 * A(a) = W_A E[a], B(b) = W_B E[b] and H(h) = W_H h under reading R1. */
void oracle_project(const uint16_t *P, int64_t rows, int64_t d, const uint16_t *x, double *out)
{
    for (int64_t r = 0; r < rows; ++r) {
        double s = 0.0;
        for (int64_t i = 0; i < d; ++i) s += bf16_to_f64(P[r * d + i]) * bf16_to_f64(x[i]);
        out[r] = s;
    }
}

/* S[i*K + j] = U[j] + sum_k A[i, k] * g[k] * B[j, k]: the pages' pair score
 * S_t(a_i, b_j) for n_prev predecessors a_i and K current candidates b_j. */
void oracle_pair_scores(int n_prev, int K, int64_t e, const double *A, const double *g,
                        const double *B, const double *U, double *S)
{
    for (int i = 0; i < n_prev; ++i)
        for (int j = 0; j < K; ++j) {
            double s = 0.0;
            for (int64_t k = 0; k < e; ++k) s += A[i * e + k] * g[k] * B[j * e + k];
            S[i * K + j] = U[j] + s;
        }
}

/* Max-sum walk (reading R3) over tables P [L, K, K]; at t = 0 only row 0 (the
 * anchor) is read. delta_0(j) = P[0,0,j];
 * delta_t(j) = max_i delta_{t-1}(i) + P[t,i,j]; backtrack from the best final
 * rank. ranks[t] is the chosen candidate rank; step_margin[t] is the gap
 * between the best and second best incoming value at the chosen node
 * (+inf at t = 0, where there is one predecessor); final_margin is the gap
 * between the best and second best delta_{L-1}. */
void oracle_viterbi(int L, int K, const double *P, int32_t *ranks, double *score,
                    double *step_margin, double *final_margin)
{
    double *delta = (double *)malloc((size_t)L * K * sizeof(double));
    double *gapm = (double *)malloc((size_t)L * K * sizeof(double));
    int32_t *bp = (int32_t *)malloc((size_t)L * K * sizeof(int32_t));
    for (int j = 0; j < K; ++j) {
        delta[j] = P[j];
        bp[j] = 0;
        gapm[j] = INFINITY;
    }
    for (int t = 1; t < L; ++t)
        for (int j = 0; j < K; ++j) {
            double best = -INFINITY, second = -INFINITY;
            int bi = -1;
            for (int i = 0; i < K; ++i) {
                double v = delta[(t - 1) * K + i] + P[((int64_t)t * K + i) * K + j];
                if (v > best) {
                    second = best;
                    best = v;
                    bi = i;
                } else if (v > second) {
                    second = v;
                }
            }
            delta[t * K + j] = best;
            bp[t * K + j] = bi;
            gapm[t * K + j] = best - second;
        }
    double best = -INFINITY, second = -INFINITY;
    int bj = -1;
    for (int j = 0; j < K; ++j) {
        double v = delta[(L - 1) * K + j];
        if (v > best) {
            second = best;
            best = v;
            bj = j;
        } else if (v > second) {
            second = v;
        }
    }
    *score = best;
    *final_margin = best - second;
    for (int t = L - 1; t >= 0; --t) {
        ranks[t] = bj;
        step_margin[t] = gapm[t * K + bj];
        bj = bp[t * K + bj];
    }
    free(delta);
    free(gapm);
    free(bp);
}

/* The literal greedy walk: from the anchor, take the best successor at each
 * step, j_t = argmax_j P[t, j_{t-1}, j] (j_{-1} = row 0). step_margin[t] is
 * the gap between the best and second best successor; the score is the sum
 * of the chosen entries. final_margin is +inf (no final choice). */
void oracle_greedy(int L, int K, const double *P, int32_t *ranks, double *score,
                   double *step_margin, double *final_margin)
{
    int prev = 0;
    double total = 0.0;
    for (int t = 0; t < L; ++t) {
        const double *row = P + ((int64_t)t * K + prev) * K;
        double best = -INFINITY, second = -INFINITY;
        int bj = -1;
        for (int j = 0; j < K; ++j) {
            if (row[j] > best) {
                second = best;
                best = row[j];
                bj = j;
            } else if (row[j] > second) {
                second = row[j];
            }
        }
        ranks[t] = bj;
        step_margin[t] = best - second;
        total += best;
        prev = bj;
    }
    *score = total;
    *final_margin = INFINITY;
}

/* Greedy verification (reading R8): n = number of leading positions where the
 * draft equals the target's argmax; emitted = draft[0..n-1], then target[n];
 * the remaining L - n entries of emitted are -1. Returns n. */
int oracle_verify(int L, const int32_t *path, const int32_t *target, int32_t *emitted)
{
    int n = 0;
    while (n < L && path[n] == target[n]) ++n;
    for (int t = 0; t < n; ++t) emitted[t] = path[t];
    emitted[n] = target[n];
    for (int t = n + 1; t <= L; ++t) emitted[t] = -1;
    return n;
}

/* Stages after top-K, for one sequence: projections, pair tables and the walk.
 * ids/vals [L, K] are the candidates and their logits. P [L, K, K] receives
 * the tables (rows 1..K-1 at t = 0 are -inf: the anchor is the only
 * predecessor there, reading R6). */
static void select_after_topk(const uint16_t *E, const uint16_t *WA, const uint16_t *WB,
                              const uint16_t *WH, int64_t d, int64_t e, int L, int K, int walk,
                              const uint16_t *h, int32_t anchor, const int32_t *ids,
                              const double *vals, double *P, int32_t *ranks, int32_t *tokens,
                              double *score, double *step_margin, double *final_margin)
{
    double *Aprev = (double *)malloc((size_t)K * e * sizeof(double));
    double *Bcur = (double *)malloc((size_t)K * e * sizeof(double));
    double *g = (double *)malloc((size_t)e * sizeof(double));
    for (int t = 0; t < L; ++t) {
        int n_prev = (t == 0) ? 1 : K;
        if (t == 0) {
            oracle_project(WA, e, d, E + (int64_t)anchor * d, Aprev);
        } else {
            for (int i = 0; i < K; ++i)
                oracle_project(WA, e, d, E + (int64_t)ids[(t - 1) * K + i] * d, Aprev + i * e);
        }
        for (int j = 0; j < K; ++j)
            oracle_project(WB, e, d, E + (int64_t)ids[t * K + j] * d, Bcur + j * e);
        oracle_project(WH, e, d, h + (int64_t)t * d, g);
        double *Pt = P + (int64_t)t * K * K;
        for (int k = 0; k < K * K; ++k) Pt[k] = -INFINITY;
        oracle_pair_scores(n_prev, K, e, Aprev, g, Bcur, vals + t * K, Pt);
    }
    if (walk == 0)
        oracle_viterbi(L, K, P, ranks, score, step_margin, final_margin);
    else
        oracle_greedy(L, K, P, ranks, score, step_margin, final_margin);
    for (int t = 0; t < L; ++t) tokens[t] = ids[t * K + ranks[t]];
    free(Aprev);
    free(Bcur);
    free(g);
}

/* The whole selector for one sequence: logits of the L positions, top-K,
 * projections, pair tables and the walk (walk 0 = Viterbi, 1 = greedy). */
void oracle_select(const uint16_t *W, const uint16_t *E, const uint16_t *WA, const uint16_t *WB,
                   const uint16_t *WH, int64_t V, int64_t d, int64_t e, int L, int K, int walk,
                   const uint16_t *h, int32_t anchor, int32_t *ids, double *vals,
                   double *topk_margin, double *P, int32_t *ranks, int32_t *tokens, double *score,
                   double *step_margin, double *final_margin, int nthreads)
{
    double *U = (double *)malloc((size_t)L * V * sizeof(double));
    oracle_logits(W, h, V, d, L, U, nthreads);
    for (int t = 0; t < L; ++t)
        oracle_topk(U + (int64_t)t * V, V, K, ids + t * K, vals + t * K, topk_margin + t);
    free(U);
    select_after_topk(E, WA, WB, WH, d, e, L, K, walk, h, anchor, ids, vals, P, ranks, tokens,
                      score, step_margin, final_margin);
}

/* The selector for one sequence with the candidate ids given (for example by
 * another implementation's top-K): their logits are recomputed here, then the
 * same projections, tables and walk as oracle_select. */
void oracle_select_given(const uint16_t *W, const uint16_t *E, const uint16_t *WA,
                         const uint16_t *WB, const uint16_t *WH, int64_t V, int64_t d, int64_t e,
                         int L, int K, int walk, const uint16_t *h, int32_t anchor,
                         const int32_t *ids, double *vals, double *P, int32_t *ranks,
                         int32_t *tokens, double *score, double *step_margin, double *final_margin)
{
    (void)V;
    for (int t = 0; t < L; ++t)
        for (int j = 0; j < K; ++j) {
            double s = 0.0;
            const uint16_t *w = W + (int64_t)ids[t * K + j] * d;
            for (int64_t i = 0; i < d; ++i) s += bf16_to_f64(w[i]) * bf16_to_f64(h[t * d + i]);
            vals[t * K + j] = s;
        }
    select_after_topk(E, WA, WB, WH, d, e, L, K, walk, h, anchor, ids, vals, P, ranks, tokens,
                      score, step_margin, final_margin);
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * Sampling (temperature T > 0). Blog "DFlash 2: Keep Drafting Parallel",
 * section "A Lightweight Path Selector": sampling draws from the same pair
 * scores, and verification by rejection sampling leaves the output distributed
 * exactly as the target's. Readings (listed in the design notes):
 *   S1  the draft distribution at step t is the softmax over the K candidate
 *       ranks of P[t, prev, .] / T, prev = the rank chosen at t-1 (row 0 at
 *       t = 0), and the step draws by inverting its CDF in rank order with a
 *       given uniform u_t: the first rank whose running sum exceeds u_t;
 *   S2  verification accepts draft token x_t with probability
 *       min(1, p_t(x_t) / q_t(x_t)) (uniform u_acc_t below it accepts); at the
 *       first rejection it draws from the residual max(0, p_t - q_t),
 *       normalised, by inverting its CDF in vocabulary order with u_res; if all
 *       L drafts are accepted it draws the bonus token from p_L the same way.
 * Uniform random numbers are inputs.
 * ------------------------------------------------------------------------- */

/* ranks [L], q_all [L, K] (the distribution drawn from at each step),
 * margin [L] = distance of u_t to the nearest CDF boundary of its step. */
void oracle_sample_walk(int L, int K, const double *P, double T, const double *u, int32_t *ranks, double *q_all,
                        double *margin)
{
    int prev = 0;
    for (int t = 0; t < L; ++t) {
        const double *row = P + ((int64_t)t * K + prev) * K;
        double m = -INFINITY;
        for (int j = 0; j < K; ++j)
            if (row[j] > m) m = row[j];
        double Z = 0.0;
        double *q = q_all + (int64_t)t * K;
        for (int j = 0; j < K; ++j) {
            q[j] = exp((row[j] - m) / T);
            Z += q[j];
        }
        for (int j = 0; j < K; ++j) q[j] /= Z;
        double c = 0.0, mg = INFINITY;
        int chosen = -1;
        for (int j = 0; j < K; ++j) {
            c += q[j];
            const double dist = fabs(c - u[t]);
            if (j < K - 1 && dist < mg) mg = dist;
            if (chosen < 0 && c > u[t]) chosen = j;
        }
        if (chosen < 0) chosen = K - 1;  /* u within rounding of 1 */
        ranks[t] = chosen;
        margin[t] = mg;
        prev = chosen;
    }
}

/* Draws from the distribution r (length V, total Z > 0) with uniform u:
 * the first index whose running sum exceeds u * Z. *margin receives the
 * smallest distance, as a fraction of Z, between u and a CDF boundary. */
static int64_t draw_inverse_cdf(const double *r, int64_t V, double u, double *margin)
{
    double Z = 0.0;
    for (int64_t y = 0; y < V; ++y) Z += r[y];
    const double target = u * Z;
    double c = 0.0, mg = INFINITY;
    int64_t chosen = -1, last = 0;
    for (int64_t y = 0; y < V; ++y) {
        if (r[y] <= 0.0) continue;
        last = y;
        c += r[y];
        const double dist = fabs(c - target) / Z;
        if (dist < mg && c < Z) mg = dist;
        if (chosen < 0 && c > target) chosen = y;
    }
    if (chosen < 0) chosen = last;
    *margin = mg;
    return chosen;
}

/* Rejection-sampling verification of one sampled draft.
 * path [L] draft tokens, ids [L, K] candidates, q [L, K] their draft
 * probabilities, p [L+1, V] target probabilities, u_acc [L], u_res.
 * Returns n (accepted drafts); emitted [L+1] = path[0..n-1], then the drawn
 * token, then -1. acc_margin[t] = |u_acc[t] - min(1, p/q)| for the decided
 * positions (+inf after the stop); res_margin = the draw's CDF margin. */
int oracle_verify_rejection(int L, int K, int64_t V, const int32_t *path, const int32_t *ids, const double *q,
                            const double *p, const double *u_acc, double u_res, int32_t *emitted,
                            double *acc_margin, double *res_margin)
{
    double *r = (double *)malloc((size_t)V * sizeof(double));
    int n = 0;
    for (int t = 0; t < L; ++t) acc_margin[t] = INFINITY;
    for (; n < L; ++n) {
        const int32_t x = path[n];
        double qx = 0.0;
        for (int j = 0; j < K; ++j)
            if (ids[n * K + j] == x) qx = q[n * K + j];
        const double px = p[(int64_t)n * V + x];
        const double a = (qx > 0.0) ? fmin(1.0, px / qx) : 0.0;
        acc_margin[n] = fabs(u_acc[n] - a);
        if (!(u_acc[n] < a)) break;
    }
    for (int t = 0; t < n; ++t) emitted[t] = path[t];
    const double *pt = p + (int64_t)n * V;
    if (n < L) {
        for (int64_t y = 0; y < V; ++y) r[y] = pt[y];
        for (int j = 0; j < K; ++j) {
            const int32_t c = ids[n * K + j];
            r[c] = fmax(0.0, pt[c] - q[n * K + j]);
        }
        double Z = 0.0;
        for (int64_t y = 0; y < V; ++y) Z += r[y];
        if (!(Z > 0.0))
            for (int64_t y = 0; y < V; ++y) r[y] = pt[y];
    } else {
        for (int64_t y = 0; y < V; ++y) r[y] = pt[y];
    }
    emitted[n] = (int32_t)draw_inverse_cdf(r, V, u_res, res_margin);
    for (int t = n + 1; t <= L; ++t) emitted[t] = -1;
    free(r);
    return n;
}

/* ---------------------------------------------------------------------------
 * Two-tap dynamic depthwise convolution. Blog "DFlash 2: Keep Drafting
 * Parallel", section "A Lightweight Local Convolution": Conv_k(x)_t =
 * k_{t,0} (.) x_t + k_{t,1} (.) x_{t-1}; each coefficient is a learned base
 * kernel plus a small correction computed from the current hidden state, and
 * every 16 channels share one correction; the first draft position reads the
 * last verified token's representation, each later one its predecessor's; nothing
 * carries over from one block to the next. Readings (listed in the design
 * notes):
 *   C1  a block is S rows: the last verified token's representation, then the
 *       draft positions; row 0 has no predecessor (x_{-1} = 0);
 *   C2  k_{t,i}[c] = base[i, c] + corr_{t,i}[c / 16], with the correction a
 *       linear map of x_t without bias: corr_{t,i}[g] = Wc[2 g + i] . x_t
 *       (Wc has 2 d/16 rows, the two taps of group g interleaved).
 * ------------------------------------------------------------------------- */

/* X [B, S, d], base [2, d], Wc [2 (d/16), d] as bf16 bits; Y [B, S, d]. */
void oracle_conv2(int64_t B, int64_t S, int64_t d, const uint16_t *X, const uint16_t *base, const uint16_t *Wc,
                  double *Y, int nthreads)
{
    const int64_t G = d / 16;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
#endif
    for (int64_t row = 0; row < B * S; ++row) {
        const int64_t t = row % S;
        const uint16_t *xt = X + row * d;
        const uint16_t *xprev = t > 0 ? xt - d : NULL;
        double *corr = (double *)malloc((size_t)(2 * G) * sizeof(double));
        for (int64_t r = 0; r < 2 * G; ++r) {
            double acc = 0.0;
            for (int64_t j = 0; j < d; ++j) acc += bf16_to_f64(Wc[r * d + j]) * bf16_to_f64(xt[j]);
            corr[r] = acc;
        }
        for (int64_t c = 0; c < d; ++c) {
            const int64_t g = c / 16;
            const double k0 = bf16_to_f64(base[c]) + corr[2 * g];
            const double k1 = bf16_to_f64(base[d + c]) + corr[2 * g + 1];
            const double prev = xprev ? bf16_to_f64(xprev[c]) : 0.0;
            Y[row * d + c] = k0 * bf16_to_f64(xt[c]) + k1 * prev;
        }
        free(corr);
    }
}
