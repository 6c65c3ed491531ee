/*
 * moe_oracle.c -- plain, slow, fp64 CPU oracle of the DeepSeek-style MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file; only the tests, the package smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or constant with the CUDA library: bf16 decoding,
 * scoring, selection, permutation and the FFN are all written out again here.
 *
 * Sources (pages, by title and section):
 *   [LLHT] "Lower latency and higher throughput with multi-node DeepSeek deployment"
 *          (Perplexity), sections "Expert Parallelism" (256 routed experts + 1 shared,
 *          8 distinct routed experts per token, weighted sum, shared output added),
 *          "MoE Router" (sort that tracks indices; per-expert aggregated routing info),
 *          "Quantization" (SiLU activation of the expert FFN).
 *   [V41]  "DeepSeek-V4.1-Flash" vLLM article, section "Kernels", Mega-Gate paragraph
 *          (gate GEMM -> expert scoring -> bias -> top-k selection).
 *   [GRACE] "GRACE-MoE" notes, section "Core Idea 1. Expert Grouping" (expert affinity
 *          matrix A built from co-activation).
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - scoring is the logistic sigmoid s = 1/(1+exp(-l)) (oracle_router_ex also offers
 *     softmax over the token's E logits, group-limited selection and unnormalised
 *     weights, the options of the other MoE families one router serves);
 *   - a group's score is the sum of its group_top largest biased scores sel;
 *   - the per-expert bias only selects: sel = s + b, the weights use the unbiased s;
 *   - order is sel descending, equal sel -> lower expert index first;
 *   - weights are renormalised over the k selected unbiased scores: w_j = s_j / sum s;
 *   - SwiGLU: h = silu(x W1) * (x W3), y = h W2, W1 being the gate projection;
 *   - the shared expert is added with weight 1;
 *   - rows of the permuted buffer are ordered by (expert asc, token asc);
 *   - affinity C[i][j] counts tokens whose top-k holds both i and j, C[i][i] = 0.
 *
 * Everything is computed in IEEE double from the exact values of the bf16 inputs,
 * with no intermediate rounding to a narrower type.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* A bf16 number is the upper half of an IEEE binary32: widen it and convert. */
static double bf16_value(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static double sigmoid(double l) { return 1.0 / (1.0 + exp(-l)); }

/* Gate GEMM and scoring for one token ([V41] Mega-Gate: gate GEMM, expert scoring, bias).
 *   l[e]   = sum_h X[t,h] * W_gate[e,h]
 *   s[e]   = sigmoid(l[e])
 *   sel[e] = s[e] + bias[e]
 */
static void score_token(const uint16_t *x, const uint16_t *Wg, const float *bias,
                        int H, int E, double *l, double *s, double *sel)
{
    for (int e = 0; e < E; ++e) {
        const uint16_t *w = Wg + (size_t)e * H;
        double acc = 0.0;
        for (int h = 0; h < H; ++h)
            acc += bf16_value(x[h]) * bf16_value(w[h]);
        l[e] = acc;
        s[e] = sigmoid(acc);
        sel[e] = s[e] + (double)bias[e];
    }
}

/* True when expert a ranks before expert b: larger sel first, lower index on ties. */
static int ranks_before(const double *sel, int a, int b)
{
    if (sel[a] != sel[b]) return sel[a] > sel[b];
    return a < b;
}

/* Softmax scoring of one token: s[e] = exp(l[e]) / sum_j exp(l[j]) over all E experts,
 * evaluated as exp(l[e] - m) / sum_j exp(l[j] - m) with m the largest logit (the same
 * value in exact arithmetic; no overflow).  sel[e] = s[e] + bias[e]. */
static void softmax_token(const double *l, const float *bias, int E, double *s, double *sel)
{
    double m = l[0];
    for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
    double sum = 0.0;
    for (int e = 0; e < E; ++e) { s[e] = exp(l[e] - m); sum += s[e]; }
    for (int e = 0; e < E; ++e) { s[e] /= sum; sel[e] = s[e] + (double)bias[e]; }
}

/* Group-limited selection ([LLHT] "MoE Router": DeepSeek routing with expert groups;
 * Mixtral's is the case of one group that holds every expert).  The E experts form
 * n_group groups of G = E / n_group consecutive experts.  A group's score is the sum of
 * its group_top largest sel; the topk_group groups with the largest score (lower group
 * index first on equal scores) stay eligible, and the experts of the other groups get
 * taken[e] = 1 so that the top-k passes over them. */
static void limit_groups(const double *sel, int E, int n_group, int topk_group, int group_top,
                         unsigned char *taken, double *gscore, unsigned char *gkeep)
{
    const int G = E / n_group;
    for (int g = 0; g < n_group; ++g) {
        /* group_top rounds of "largest sel of the group not yet counted" */
        double sum = 0.0;
        for (int r = 0; r < group_top; ++r) {
            int best = -1;
            for (int e = g * G; e < (g + 1) * G; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ranks_before(sel, e, best)) best = e;
            }
            taken[best] = 1;
            sum += sel[best];
        }
        for (int e = g * G; e < (g + 1) * G; ++e) taken[e] = 0;
        gscore[g] = sum;
        gkeep[g] = 0;
    }
    for (int r = 0; r < topk_group; ++r) {
        int best = -1;
        for (int g = 0; g < n_group; ++g) {
            if (gkeep[g]) continue;
            if (best < 0 || gscore[g] > gscore[best]) best = g;   /* ties: lower g stays */
        }
        gkeep[best] = 1;
    }
    for (int e = 0; e < E; ++e) taken[e] = gkeep[e / G] ? 0 : 1;
}

/* Top-k for one token ([LLHT] "MoE Router": a sort that keeps the indices): k rounds of
 * "take the best expert not yet taken" over the experts with taken[e] == 0 (the others
 * are skipped); the result is in rank order. */
static void topk_eligible(const double *sel, int E, int K, int32_t *idx, unsigned char *taken)
{
    for (int j = 0; j < K; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            if (best < 0 || ranks_before(sel, e, best)) best = e;
        }
        taken[best] = 1;
        idx[j] = best;
    }
}

/* Router with the routing options of one MoE family:
 *   scoring     0: s = sigmoid(l) ([V41] Mega-Gate);  1: s = softmax of the token's E logits
 *   n_group, topk_group, group_top: group-limited selection (limit_groups); n_group = 1
 *               selects over all experts
 *   renorm      1: w_j = s_j / sum of the K selected s ([V41]; the bias never enters the
 *               weights);  0: w_j = s_j
 * Outputs as oracle_router.  Returns -1 on arguments that do not define a selection. */
int oracle_router_ex(const uint16_t *X, const uint16_t *Wg, const float *bias,
                     int T, int H, int E, int K, int scoring, int n_group, int topk_group,
                     int group_top, int renorm, int32_t *topk_idx, double *topk_w,
                     double *logits, double *scores, double *sel_out)
{
    if (T < 0 || H <= 0 || E <= 0 || K <= 0 || K > E) return -1;
    if (scoring != 0 && scoring != 1) return -1;
    if (n_group < 1 || E % n_group != 0 || topk_group < 1 || topk_group > n_group) return -1;
    if (group_top < 1 || group_top > E / n_group || K > topk_group * (E / n_group)) return -1;
#pragma omp parallel
    {
        double *l = (double *)malloc(sizeof(double) * (size_t)E);
        double *s = (double *)malloc(sizeof(double) * (size_t)E);
        double *sel = (double *)malloc(sizeof(double) * (size_t)E);
        double *gscore = (double *)malloc(sizeof(double) * (size_t)n_group);
        unsigned char *gkeep = (unsigned char *)malloc((size_t)n_group);
        unsigned char *taken = (unsigned char *)malloc((size_t)E);
#pragma omp for schedule(dynamic, 4)
        for (int t = 0; t < T; ++t) {
            score_token(X + (size_t)t * H, Wg, bias, H, E, l, s, sel);
            if (scoring == 1) softmax_token(l, bias, E, s, sel);
            int32_t *idx = topk_idx + (size_t)t * K;
            memset(taken, 0, (size_t)E);
            if (n_group > 1) limit_groups(sel, E, n_group, topk_group, group_top, taken, gscore, gkeep);
            topk_eligible(sel, E, K, idx, taken);
            /* weights from the selected, unbiased scores */
            double denom = 0.0;
            for (int j = 0; j < K; ++j) denom += s[idx[j]];
            for (int j = 0; j < K; ++j)
                topk_w[(size_t)t * K + j] = renorm ? s[idx[j]] / denom : s[idx[j]];
            if (logits) memcpy(logits + (size_t)t * E, l, sizeof(double) * (size_t)E);
            if (scores) memcpy(scores + (size_t)t * E, s, sizeof(double) * (size_t)E);
            if (sel_out) memcpy(sel_out + (size_t)t * E, sel, sizeof(double) * (size_t)E);
        }
        free(l); free(s); free(sel); free(gscore); free(gkeep); free(taken);
    }
    return 0;
}

/* Router: sigmoid scores, top-k over all experts and renormalised weights for every token.
 *   topk_idx[T,K] int32 (rank order), topk_w[T,K] double,
 *   logits/scores/sel[T,E] double, each nullable. */
int oracle_router(const uint16_t *X, const uint16_t *Wg, const float *bias,
                  int T, int H, int E, int K,
                  int32_t *topk_idx, double *topk_w,
                  double *logits, double *scores, double *sel_out)
{
    return oracle_router_ex(X, Wg, bias, T, H, E, K, 0, 1, 1, 1, 1, topk_idx, topk_w, logits,
                            scores, sel_out);
}

/* Dispatch bookkeeping ([LLHT] "MoE Router": per-expert aggregated routing info;
 * "Expert Parallelism": tokens are sent to their experts before the expert GEMMs).
 *   counts[e]      = number of (t,j) with topk_idx[t,j] == e
 *   offsets[e]     = counts[0] + ... + counts[e-1], offsets[E] = T*K
 *   perm[r]        = token of permuted row r, rows ordered by (expert, token)
 *   slot_pos[t,j]  = permuted row that holds (t, j)
 *   affinity[i,j]  = tokens whose top-k holds both i and j (i != j), 0 on the diagonal
 *                    ([GRACE] expert affinity matrix A); nullable. */
int oracle_dispatch(const int32_t *topk_idx, int T, int E, int K,
                    int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *slot_pos,
                    int32_t *affinity)
{
    if (T < 0 || E <= 0 || K <= 0) return -1;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (size_t i = 0; i < (size_t)T * K; ++i) {
        int e = topk_idx[i];
        if (e < 0 || e >= E) return -2;
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];

    /* stable counting sort: walk experts in order, tokens in order inside each expert */
    int32_t r = 0;
    for (int e = 0; e < E; ++e)
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < K; ++j)
                if (topk_idx[(size_t)t * K + j] == e) {
                    perm[r] = t;
                    slot_pos[(size_t)t * K + j] = r;
                    ++r;
                }

    if (affinity) {
        memset(affinity, 0, sizeof(int32_t) * (size_t)E * E);
        for (int t = 0; t < T; ++t) {
            const int32_t *idx = topk_idx + (size_t)t * K;
            for (int a = 0; a < K; ++a)
                for (int b = 0; b < K; ++b)
                    if (a != b) affinity[(size_t)idx[a] * E + idx[b]] += 1;
        }
    }
    return 0;
}

/* One expert applied to one token row ([LLHT] "Quantization": SiLU activation of the
 * expert MLP; "SiLU and multiply"):
 *   u = x W1, v = x W3          (W1, W3 are [H, I], I contiguous)
 *   h = silu(u) * v = u / (1 + exp(-u)) * v
 *   y = h W2                    (W2 is [I, H], H contiguous)
 * u, v, h are kept in double; nothing is rounded between the steps. */
static void expert_row(const uint16_t *x, const uint16_t *W1, const uint16_t *W3,
                       const uint16_t *W2, int H, int I, double *u, double *v, double *y)
{
    for (int i = 0; i < I; ++i) { u[i] = 0.0; v[i] = 0.0; }
    for (int h = 0; h < H; ++h) {
        double xh = bf16_value(x[h]);
        const uint16_t *w1 = W1 + (size_t)h * I;
        const uint16_t *w3 = W3 + (size_t)h * I;
        for (int i = 0; i < I; ++i) {
            u[i] += xh * bf16_value(w1[i]);
            v[i] += xh * bf16_value(w3[i]);
        }
    }
    for (int i = 0; i < I; ++i) u[i] = u[i] / (1.0 + exp(-u[i])) * v[i]; /* u now holds h */
    for (int c = 0; c < H; ++c) y[c] = 0.0;
    for (int i = 0; i < I; ++i) {
        const uint16_t *w2 = W2 + (size_t)i * H;
        for (int c = 0; c < H; ++c) y[c] += u[i] * bf16_value(w2[c]);
    }
}

/* Expert FFN of individual rows: y[n,:] = FFN_e(x_n) with the expert weights passed in
 * per row (W1[n], W3[n], W2[n] point at that row's expert).  x rows are [H] bf16. */
int oracle_expert_rows(const uint16_t *const *xrows, const uint16_t *const *W1,
                       const uint16_t *const *W3, const uint16_t *const *W2,
                       int n, int H, int I, double *y)
{
    if (n < 0 || H <= 0 || I <= 0) return -1;
#pragma omp parallel
    {
        double *u = (double *)malloc(sizeof(double) * (size_t)I);
        double *v = (double *)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n; ++r)
            expert_row(xrows[r], W1[r], W3[r], W2[r], H, I, u, v, y + (size_t)r * H);
        free(u); free(v);
    }
    return 0;
}

/* Full layer output for a list of tokens ([LLHT] "Expert Parallelism": each token goes
 * to k distinct routed experts whose results are summed with the routing weights, and
 * the shared expert's result is added):
 *   Y[t] = sum_j topk_w[t,j] * FFN_{topk_idx[t,j]}(X[t]) + FFN_shared(X[t])
 * Routed expert weights are addressed per expert (W1e[e] -> [H,I] etc.); an expert that
 * no listed token uses may be NULL.  Is == 0 means no shared expert.
 * tokens[n] are token indices into X / topk_*; Y is [n, H] double. */
int oracle_layer_tokens(const uint16_t *X, int H, int I, int Is, int K,
                        const int32_t *topk_idx, const double *topk_w,
                        const uint16_t *const *W1e, const uint16_t *const *W3e,
                        const uint16_t *const *W2e,
                        const uint16_t *W1s, const uint16_t *W3s, const uint16_t *W2s,
                        const int32_t *tokens, int n, double *Y)
{
    if (n < 0 || H <= 0 || I <= 0 || K <= 0 || Is < 0) return -1;
    for (int q = 0; q < n; ++q)
        for (int j = 0; j < K; ++j)
            if (!W1e[topk_idx[(size_t)tokens[q] * K + j]]) return -3;
    int Imax = I > Is ? I : Is;
    int rc = 0;
#pragma omp parallel
    {
        double *u = (double *)malloc(sizeof(double) * (size_t)Imax);
        double *v = (double *)malloc(sizeof(double) * (size_t)Imax);
        double *ye = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
        for (int q = 0; q < n; ++q) {
            int t = tokens[q];
            const uint16_t *x = X + (size_t)t * H;
            double *y = Y + (size_t)q * H;
            for (int c = 0; c < H; ++c) y[c] = 0.0;
            for (int j = 0; j < K; ++j) {
                int e = topk_idx[(size_t)t * K + j];
                double w = topk_w[(size_t)t * K + j];
                expert_row(x, W1e[e], W3e[e], W2e[e], H, I, u, v, ye);
                for (int c = 0; c < H; ++c) y[c] += w * ye[c];
            }
            if (Is > 0) {
                expert_row(x, W1s, W3s, W2s, H, Is, u, v, ye);
                for (int c = 0; c < H; ++c) y[c] += ye[c];
            }
        }
        free(u); free(v); free(ye);
    }
    return rc;
}

/* Combine on its own ([LLHT] "Expert Parallelism": weighted sum of the routed results,
 * shared result added):  Y[t] = sum_j topk_w[t,j] * Yp[slot_pos[t,j]] (+ Ysh[t]).
 * Yp is bf16 [rows, H], Ysh is double [T, H] or NULL, Y is double [T, H]. */
int oracle_combine(const uint16_t *Yp, const int32_t *slot_pos, const double *topk_w,
                   const double *Ysh, int T, int H, int K, double *Y)
{
    if (T < 0 || H <= 0 || K <= 0) return -1;
    for (int t = 0; t < T; ++t) {
        double *y = Y + (size_t)t * H;
        for (int c = 0; c < H; ++c) y[c] = 0.0;
        for (int j = 0; j < K; ++j) {
            const uint16_t *row = Yp + (size_t)slot_pos[(size_t)t * K + j] * H;
            double w = topk_w[(size_t)t * K + j];
            for (int c = 0; c < H; ++c) y[c] += w * bf16_value(row[c]);
        }
        if (Ysh)
            for (int c = 0; c < H; ++c) y[c] += Ysh[(size_t)t * H + c];
    }
    return 0;
}

/* Number of threads the OpenMP runtime will use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the calling thread's later oracle calls (n >= 1); returns the previous
 * count.  For timing the oracle on one core beside all of them. */
int oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    const int prev = omp_get_max_threads();
    if (n >= 1) omp_set_num_threads(n);
    return prev;
#else
    (void)n;
    return 1;
#endif
}
