/*
 * moe_oracle.c -- plain, slow, CPU reference of the MoE tree-verification layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library. It shares no code, header
 * or table with the CUDA path, and the CUDA path never calls it.
 *
 * Sources (page title + section):
 *   [LAYER]  "MoE and speculative decoding: joint optimisation of compute,
 *            communication and acceptance" (blog), section "starting from one MoE
 *            layer": E(x) = TopR(softmax(W_r x)), y = sum_{e in E(x)} g_e(x) E_e(x),
 *            and the router -> permute/group -> grouped GEMM -> unpermute+combine
 *            pipeline.
 *   [UNION]  same blog, section "dense vs MoE verification": the working set of a
 *            verification is the union of the experts chosen by its tokens.
 *   [ACCEPT] "AcceptMoE" news article, section 02: commitment probability per draft
 *            position weights the target router scores; the root node's natural
 *            top-k is kept (root anchor); the set size follows the effective rank of
 *            the demand distribution; residency-aware pruning removes low-demand
 *            non-resident experts within a rerouting budget and a minimum set size.
 *   [ECO]    "Fewer experts, faster decoding: cost-aware speculative decoding for MoE"
 *            (EcoSpec, arXiv 2607.12696), abstract, section 1 and Fig. 2-3: before
 *            verification, choose the candidate nodes greedily by acceptance likelihood
 *            minus a weight times the number of new predicted experts, tracking the
 *            experts the chosen nodes already cover in a buffer. The same scoring rule is
 *            written out in the "MoE and speculative decoding" blog as
 *            Score(v) = log P_q(v) - lambda * dC_expert(v).
 *   [ABS]    AcceptMoE abstract (arXiv 2608.02989): a verifier-side selector that
 *            combines target-router scores with offline commitment probabilities,
 *            sizes the eligible set per verification block, and constrains
 *            target-expert eligibility (re-route inside the eligible set).
 *
 * The pages give the method in prose only. Where a step is left open, the reading
 * taken is stated at the step (demand D_e = sum_n c(depth_n) softmax(l_n)_e,
 * m = max(k, ceil(exp H)) capped at the pool size, pool = natural union, prune in
 * ascending demand with a count budget, gates renormalised over the chosen k).
 *
 * Precision: every floating-point step runs in fp64 on inputs upcast exactly from
 * fp32/bf16. Decisions that compare router logits (top-k) take them in fp32, the
 * precision the logits have on the device, so both sides decide on equal values.
 *
 * Parity unpinned: the exact integer rounding of exp(H) and the candidate-pool rule
 * used by the AcceptMoE authors (the pages print no worked selection example).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

enum { ORC_NATURAL = 0, ORC_ACCEPT = 1, ORC_FIXED_B = 2 };

/* bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 word. */
static double elem(const void *p, int dtype, size_t i) {
    if (dtype == 0) return (double)((const float *)p)[i];
    uint32_t u = ((uint32_t)((const uint16_t *)p)[i]) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Nearest bf16 to v, ties to the even significand, as raw bits. bf16 keeps 8
 * significant bits and fp32's exponent range: normal numbers from 2^-126, subnormals in
 * steps of 2^-133, largest finite (2 - 2^-7) * 2^127. Written from that definition:
 * v = m * 2^e with 1/2 <= |m| < 1, so the quantum at v is 2^(e-8) (never below 2^-133);
 * nearbyint rounds to nearest even in the default rounding mode. */
ORC_API uint16_t oracle_round_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    const uint16_t sign = signbit(v) ? 0x8000 : 0;
    const double a = fabs(v);
    double r;
    if (a == 0.0 || isinf(a)) {
        r = a;
    } else {
        int e;
        frexp(a, &e);
        int qexp = e - 8;
        if (qexp < -133) qexp = -133;
        r = ldexp(nearbyint(ldexp(a, -qexp)), qexp);
        if (r > ldexp(255.0, 120)) r = INFINITY; /* past (2 - 2^-7) * 2^127 */
    }
    /* r is a bf16 value (or inf), so it is exact in fp32 and its low 16 bits are 0 */
    const float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* Pre-norm of the layer input (the RMS normalisation the target models put in front of
 * the MoE layer, without a learned weight): xn[r, i] = x[r, i] / sqrt(mean_i x[r, i]^2 +
 * eps), all in fp64, each element then rounded once to the input dtype (nearest, ties
 * to even). xn64 [R, d] (may be NULL) receives the values before that rounding. */
ORC_API void oracle_rmsnorm(const void *x, int dtype, int R, int d, double eps, double *xn64,
                            void *xn) {
    for (int n = 0; n < R; ++n) {
        double ss = 0.0;
        for (int i = 0; i < d; ++i) {
            const double v = elem(x, dtype, (size_t)n * d + i);
            ss += v * v;
        }
        const double scale = 1.0 / sqrt(ss / d + eps);
        for (int i = 0; i < d; ++i) {
            const size_t at = (size_t)n * d + i;
            const double v = elem(x, dtype, at) * scale;
            if (xn64) xn64[at] = v;
            if (dtype == 0)
                ((float *)xn)[at] = (float)v;
            else
                ((uint16_t *)xn)[at] = oracle_round_bf16(v);
        }
    }
}

/* [LAYER] router scores l = W_r x, one row per token; no bias. */
ORC_API void oracle_router(const void *x, const void *Wr, int dtype, int R, int d, int E,
                           double *logits) {
    for (int n = 0; n < R; ++n)
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int i = 0; i < d; ++i)
                s += elem(x, dtype, (size_t)n * d + i) * elem(Wr, dtype, (size_t)e * d + i);
            logits[(size_t)n * E + e] = s;
        }
}

/* [LAYER] TopR: the k largest scores of one row, in descending order, ties to the
 * lower expert id. softmax is monotone, so top-k of the probabilities is top-k of
 * the logits. `allowed` (may be NULL) restricts the candidates. Returns the smallest
 * gap between consecutive scores among the k chosen and the best score left out (the
 * order of the k is part of the result), +inf if there is no such pair. */
static double topk_row(const float *l, int E, int k, const unsigned char *allowed, int *out) {
    unsigned char taken[1024];
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if ((allowed && !allowed[e]) || taken[e]) continue;
            if (best < 0 || l[e] > l[best]) best = e;
        }
        out[j] = best;
        if (best >= 0) taken[best] = 1;
    }
    int rest = -1;
    for (int e = 0; e < E; ++e) {
        if ((allowed && !allowed[e]) || taken[e]) continue;
        if (rest < 0 || l[e] > l[rest]) rest = e;
    }
    double gap = INFINITY;
    for (int j = 0; j + 1 < k; ++j)
        if (out[j + 1] >= 0 && (double)l[out[j]] - (double)l[out[j + 1]] < gap)
            gap = (double)l[out[j]] - (double)l[out[j + 1]];
    if (rest >= 0 && out[k - 1] >= 0 && (double)l[out[k - 1]] - (double)l[rest] < gap)
        gap = (double)l[out[k - 1]] - (double)l[rest];
    return gap;
}

ORC_API double oracle_topk(const float *logits, int R, int E, int k, int *idx) {
    double margin = INFINITY;
    for (int n = 0; n < R; ++n) {
        double g = topk_row(logits + (size_t)n * E, E, k, NULL, idx + (size_t)n * k);
        if (g < margin) margin = g;
    }
    return margin;
}

/* softmax of one row of fp32 logits in fp64: exp(l_e - max) / sum_e' exp(l_e' - max),
 * the sum taken in ascending expert order. */
static void softmax_row(const float *l, int E, double *p) {
    double mx = l[0], s = 0.0;
    for (int e = 1; e < E; ++e)
        if (l[e] > mx) mx = l[e];
    for (int e = 0; e < E; ++e) {
        p[e] = exp((double)l[e] - mx);
        s += p[e];
    }
    for (int e = 0; e < E; ++e) p[e] /= s;
}

/* Fill order: a before b when D_a > D_b, or equal demand and lower id. */
static int before_desc(const double *D, int a, int b) {
    return D[a] > D[b] || (D[a] == D[b] && a < b);
}

/* Pruning order: a before b when D_a < D_b, or equal demand and lower id. */
static int before_asc(const double *D, int a, int b) {
    return D[a] < D[b] || (D[a] == D[b] && a < b);
}

/* exp(H) within this relative distance of an integer counts as that integer: the
 * effective rank of a demand that is exactly uniform over j experts is exactly j, but
 * evaluating it rounds to j(1 +- a few 1e-16); 1e-9 lies far above that fp64 noise and
 * far below any distance a real tree's demand produces. */
#define SNAP 1e-9

/* The set size the effective rank r asks for: the integer n when r is within SNAP*r of
 * it, else ceil(r); then floored at k and capped at the pool size. */
static int size_from_rank(double r, int k, int pool) {
    const double rn = nearbyint(r);
    int m = (fabs(r - rn) <= SNAP * r) ? (int)rn : (int)ceil(r);
    if (m < k) m = k;
    if (m > pool) m = pool;
    return m;
}

/* Relative distance of r to the nearest value where size_from_rank changes. Below an
 * integer n the size is n all the way up to the integer; it becomes n + 1 once r is more
 * than SNAP*r above n, i.e. at b_n = n / (1 - SNAP). A b_n counts only where the floor
 * and the cap leave n and n + 1 distinct. +inf if no b_n is within one unit of r. */
static double rank_margin(double r, int k, int pool) {
    double best = INFINITY;
    const double nf = floor(r);
    for (double n = nf - 1.0; n <= nf + 1.0; n += 1.0) {
        if (n < 1.0) continue;
        const int lo = n < k ? k : (n > pool ? pool : (int)n);
        const int hi = n + 1.0 < k ? k : (n + 1.0 > pool ? pool : (int)n + 1);
        if (lo == hi) continue;
        const double b = n / (1.0 - SNAP);
        const double g = fabs(r - b) / r;
        if (g < best) best = g;
    }
    return best;
}

/* Step 6 for one node: its k best logits inside the eligible set (`allowed`; NULL = all
 * experts), in descending order, ties to the lower id, and the gates: the softmax over the
 * k chosen logits (fp64, from the fp32 logits). Returns topk_row's gap. */
static double route_row(const float *l, int E, int k, const unsigned char *allowed, int *o,
                        double *g) {
    const double gap = topk_row(l, E, k, allowed, o);
    const double mx = l[o[0]];
    double s = 0.0;
    for (int j = 0; j < k; ++j) {
        g[j] = exp((double)l[o[j]] - mx);
        s += g[j];
    }
    for (int j = 0; j < k; ++j) g[j] /= s;
    return gap;
}

/* [ABS] re-routing inside an eligible set, on its own: route_row for R rows with one
 * eligibility mask (allowed [E], nonzero = eligible; it must hold at least k experts). */
ORC_API void oracle_restricted_route(const float *logits, int R, int E, int k,
                                     const unsigned char *allowed, int *idx, double *gates) {
    for (int n = 0; n < R; ++n)
        route_row(logits + (size_t)n * E, E, k, allowed, idx + (size_t)n * k,
                  gates + (size_t)n * k);
}

/* Selection for one draft tree of N nodes (node 0 is the root).
 *
 * Steps ([ACCEPT] + [ABS]):
 *  1. natural top-k per node; natural union U.
 *  2. demand D_e = sum_n c(depth_n) * softmax(l_n)_e, nodes in ascending order;
 *     c(depth) beyond the table repeats the last entry.
 *  3. effective rank r = exp(H(D / sum D)), H = -sum q ln q over all E experts.
 *     m = max(k, ceil(r)) (a value within 1e-9 relative of an integer counts as that
 *     integer), capped at the pool size. FIXED_B takes m = max(k, fixed_B) instead.
 *  4. root anchor A = natural top-k of node 0 (when `anchor`); S = A plus the best
 *     m - |A| experts of pool \ A in (D desc, id asc) order. pool = U, or all experts.
 *  5. residency-aware pruning (when `prune`): members of S \ A that are not resident
 *     are removed in (D asc, id asc) order while fewer than `budget` have been
 *     removed and |S| > max(min_set, k).
 *  6. restricted top-k: each node takes its k best logits inside S, gates are the
 *     softmax over the k chosen logits. NATURAL: S = all experts.
 *
 * Steps 2-3 run in fp64 (softmax, demand, entropy, exp).
 *
 * info[0..3] = |U|, |union of restricted choices|, |S| after step 4 (m), removed.
 * margins[0] = smallest top-k gap (fp32 logits, natural), margins[1] = relative
 * distance of r to the nearest value where the size rule changes m (rank_margin),
 * margins[2] = relative demand gap at the fill cut, margins[3] = relative demand gap
 * at the prune cut, margins[4] = smallest restricted top-k gap; +inf where a decision
 * does not depend on the demand. *r_out = r (NaN outside ACCEPT mode). Returns 0, or -1
 * on bad arguments. */
ORC_API int oracle_select_tree(const float *logits, const int *depth, int N, int E, int k,
                               const double *c, int n_c, int mode, int pool_all, int anchor,
                               int prune, const unsigned char *resident, int budget,
                               int min_set, int fixed_B, int *idx, double *gates,
                               unsigned char *eligible, int *info, double *D, double *margins,
                               double *r_out) {
    if (N < 1 || E < 1 || E > 1024 || k < 1 || k > E || n_c < 1) return -1;
    int *nat = (int *)malloc(sizeof(int) * (size_t)N * k);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    unsigned char inU[1024], inS[1024], inA[1024];
    for (int m = 0; m < 5; ++m) margins[m] = INFINITY;
    *r_out = NAN;

    /* 1. natural top-k and union */
    memset(inU, 0, (size_t)E);
    for (int n = 0; n < N; ++n) {
        double g = topk_row(logits + (size_t)n * E, E, k, NULL, nat + (size_t)n * k);
        if (g < margins[0]) margins[0] = g;
        for (int j = 0; j < k; ++j) inU[nat[(size_t)n * k + j]] = 1;
    }
    int U = 0;
    for (int e = 0; e < E; ++e) U += inU[e];
    info[0] = U;
    info[3] = 0;

    if (mode == ORC_NATURAL) {
        memset(inS, 1, (size_t)E);
        info[2] = E;
    } else {
        /* 2. commitment-weighted demand, 3. effective rank and set size */
        int pool = pool_all ? E : U;
        for (int e = 0; e < E; ++e) D[e] = 0.0;
        for (int n = 0; n < N; ++n) {
            int t = depth[n] < n_c ? depth[n] : n_c - 1;
            softmax_row(logits + (size_t)n * E, E, p);
            for (int e = 0; e < E; ++e) D[e] += c[t] * p[e];
        }
        int m;
        if (mode == ORC_ACCEPT) {
            double sum = 0.0, H = 0.0;
            for (int e = 0; e < E; ++e) sum += D[e];
            for (int e = 0; e < E; ++e) {
                double q = D[e] / sum;
                if (q > 0.0) H -= q * log(q);
            }
            const double r = exp(H);
            *r_out = r;
            m = size_from_rank(r, k, pool);
            margins[1] = rank_margin(r, k, pool);
        } else {
            m = fixed_B;
            if (m < k) m = k;
            if (m > pool) m = pool;
        }
        /* 4. anchor + fill */
        memset(inA, 0, (size_t)E);
        memset(inS, 0, (size_t)E);
        int size = 0;
        if (anchor)
            for (int j = 0; j < k; ++j) {
                inA[nat[j]] = 1;
                inS[nat[j]] = 1;
            }
        for (int e = 0; e < E; ++e) size += inS[e];
        int last = -1;
        while (size < m) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (inS[e] || !(pool_all || inU[e])) continue;
                if (best < 0 || before_desc(D, e, best)) best = e;
            }
            inS[best] = 1;
            last = best;
            ++size;
        }
        if (last >= 0) {
            int next = -1;
            for (int e = 0; e < E; ++e) {
                if (inS[e] || !(pool_all || inU[e])) continue;
                if (next < 0 || before_desc(D, e, next)) next = e;
            }
            if (next >= 0) margins[2] = (D[last] - D[next]) / D[last];
        }
        info[2] = size;
        /* 5. residency-aware pruning */
        if (prune && resident) {
            int floor_ = min_set > k ? min_set : k;
            int removed = 0, lastr = -1;
            for (;;) {
                int worst = -1;
                for (int e = 0; e < E; ++e) {
                    if (!inS[e] || inA[e] || resident[e]) continue;
                    if (worst < 0 || before_asc(D, e, worst)) worst = e;
                }
                if (worst < 0) break;
                if (removed >= budget || size <= floor_) {
                    if (lastr >= 0) margins[3] = (D[worst] - D[lastr]) / D[worst];
                    break;
                }
                inS[worst] = 0;
                --size;
                ++removed;
                lastr = worst;
            }
            info[3] = removed;
        }
    }

    /* 6. restricted top-k and renormalised gates */
    memset(inU, 0, (size_t)E);
    for (int n = 0; n < N; ++n) {
        int *o = idx + (size_t)n * k;
        double g = route_row(logits + (size_t)n * E, E, k, inS, o, gates + (size_t)n * k);
        if (g < margins[4]) margins[4] = g;
        for (int j = 0; j < k; ++j) inU[o[j]] = 1;
    }
    int Us = 0;
    for (int e = 0; e < E; ++e) Us += inU[e];
    info[1] = Us;
    for (int e = 0; e < E; ++e) eligible[e] = inS[e];
    free(nat);
    free(p);
    return 0;
}

/* [LAYER] permute / group by expert: a stable counting sort of the assignments
 * (row r, slot j) -> expert idx[r*k+j] with key (expert, row, slot). counts[e] is the
 * number of assignments of expert e, offsets[e] its exclusive prefix (offsets[E] =
 * R*k), perm[p] the assignment id r*k+j at permuted position p. */
ORC_API void oracle_permute(const int *idx, int R, int k, int E, int *counts, int *offsets,
                            int *perm) {
    int *cur = (int *)calloc((size_t)E, sizeof(int));
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int a = 0; a < R * k; ++a) counts[idx[a]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    for (int r = 0; r < R; ++r)
        for (int j = 0; j < k; ++j) {
            int e = idx[r * k + j];
            perm[offsets[e] + cur[e]++] = r * k + j;
        }
    free(cur);
}

/* [LAYER] one routed expert E_e(x) as a SwiGLU FFN:
 *   a = W_gate[e] x, b = W_up[e] x, h = silu(a) * b, out = W_down[e] h,
 * silu(a) = a / (1 + exp(-a)). W_gate, W_up are [E, f, d]; W_down is [E, d, f]. */
ORC_API void oracle_expert_ffn(const double *x, int e, const void *Wg, const void *Wu,
                               const void *Wd, int dtype, int d, int f, double *out) {
    double *h = (double *)malloc(sizeof(double) * (size_t)f);
    size_t base_gu = (size_t)e * f * d, base_d = (size_t)e * d * f;
    for (int i = 0; i < f; ++i) {
        double a = 0.0, b = 0.0;
        for (int t = 0; t < d; ++t) {
            a += elem(Wg, dtype, base_gu + (size_t)i * d + t) * x[t];
            b += elem(Wu, dtype, base_gu + (size_t)i * d + t) * x[t];
        }
        h[i] = a / (1.0 + exp(-a)) * b;
    }
    for (int t = 0; t < d; ++t) {
        double s = 0.0;
        for (int i = 0; i < f; ++i) s += elem(Wd, dtype, base_d + (size_t)t * f + i) * h[i];
        out[t] = s;
    }
    free(h);
}

/* [LAYER] y_r = sum_j g_{r,j} E_{idx_{r,j}}(x_r), slots in ascending order, for the
 * rows listed in `rows` (all R rows when rows == NULL). y is [n_rows, d]. */
ORC_API void oracle_moe_combine(const void *x, const void *Wg, const void *Wu, const void *Wd,
                                int dtype, int d, int f, const int *idx, const double *gates,
                                int k, const int *rows, int n_rows, double *y) {
    double *xr = (double *)malloc(sizeof(double) * (size_t)d);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    for (int q = 0; q < n_rows; ++q) {
        int r = rows ? rows[q] : q;
        for (int t = 0; t < d; ++t) xr[t] = elem(x, dtype, (size_t)r * d + t);
        double *yr = y + (size_t)q * d;
        for (int t = 0; t < d; ++t) yr[t] = 0.0;
        for (int j = 0; j < k; ++j) {
            oracle_expert_ffn(xr, idx[(size_t)r * k + j], Wg, Wu, Wd, dtype, d, f, o);
            double g = gates[(size_t)r * k + j];
            for (int t = 0; t < d; ++t) yr[t] += g * o[t];
        }
    }
    free(xr);
    free(o);
}

/* [ECO] cost-aware draft selection. Candidates 0..C-1, node 0 the root, parent[v] < v;
 * logp[v] the cumulative draft log-probability; footprint[v*k .. v*k+k) the experts the
 * node is predicted to use. The cost term is the size of a set difference, so an id
 * listed twice in one footprint counts once, and ids outside [0, E) name no expert and
 * are skipped. S starts as {root} and the buffer B as its footprint; then, gamma - 1
 * times, among the candidates not in S whose parent is in S, take the one with the
 * largest score logp[v] - lambda * |footprint(v) \ B| (computed in fp32: one product,
 * one difference; ties to the lower index), and add it to S and its footprint to B.
 * selected[] receives S in selection order (every parent before its children),
 * *n_union = |B|. Returns the number selected (< gamma when the tree has fewer
 * candidates). */
static void add_footprint(const int *f, int k, int E, unsigned char *inB) {
    for (int j = 0; j < k; ++j)
        if (f[j] >= 0 && f[j] < E) inB[f[j]] = 1;
}

/* |f \ B| over the distinct valid ids of f */
static int new_experts(const int *f, int k, int E, const unsigned char *inB) {
    int dc = 0;
    for (int j = 0; j < k; ++j) {
        if (f[j] < 0 || f[j] >= E || inB[f[j]]) continue;
        int seen = 0;
        for (int i = 0; i < j; ++i) seen |= f[i] == f[j];
        dc += !seen;
    }
    return dc;
}

ORC_API int oracle_draft_select(int C, int k, int E, const int *parent, const float *logp,
                                const int *footprint, float lambda, int gamma, int *selected,
                                int *n_union) {
    unsigned char *inS = (unsigned char *)calloc((size_t)(C > 0 ? C : 1), 1);
    unsigned char *inB = (unsigned char *)calloc((size_t)(E > 0 ? E : 1), 1);
    int n = 0;
    if (C < 1 || gamma < 1) {
        *n_union = 0;
        free(inS);
        free(inB);
        return 0;
    }
    inS[0] = 1;
    selected[n++] = 0;
    add_footprint(footprint, k, E, inB);
    while (n < gamma) {
        int best = -1;
        float best_sc = 0.f;
        for (int v = 1; v < C; ++v) {
            if (inS[v] || parent[v] < 0 || parent[v] >= C || !inS[parent[v]]) continue;
            const int dc = new_experts(footprint + (size_t)v * k, k, E, inB);
            const float pen = lambda * (float)dc;
            const float sc = logp[v] - pen;
            if (best < 0 || sc > best_sc) {
                best = v;
                best_sc = sc;
            }
        }
        if (best < 0) break;
        inS[best] = 1;
        selected[n++] = best;
        add_footprint(footprint + (size_t)best * k, k, E, inB);
    }
    int u = 0;
    for (int e = 0; e < E; ++e) u += inB[e];
    *n_union = u;
    free(inS);
    free(inB);
    return n;
}
