/*
 * moe_oracle.c -- TEST INFRASTRUCTURE, not product code.
 *
 * The plain, slow fp64 CPU oracle for the forward pass of a Mixture-of-Experts
 * SwiGLU FFN layer.  Only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only in the seeded inputs that the
 * test harness hands to both.
 *
 * Every floating-point step is done in IEEE double from the exact stored input
 * values (fp32, or bf16 widened exactly), with no intermediate rounding to a
 * narrower type.  Loops are written in the per-token form that the pages use as
 * the definition of the layer; nothing is blocked, fused or reordered beyond an
 * OpenMP split over independent tokens.
 *
 * Sources, by page title and section:
 *  [MoE-Arch]   "MoE Architecture" (infra.bea.ai), section 2 "The Router" /
 *               "Gating Function" and "Load Balancing"; section 3 "Shared
 *               Experts"; section 1 "The Core Idea" (y = sum_i g_i Expert_i(x)).
 *  [MoE-Notes]  "Mixture of Experts" (avinashkadimisetty.com notes), "How it
 *               works": routing math g(x) = softmax(W_g x), keep top-k and
 *               renormalise "in many implementations"; capacity and dropping.
 *  [Handbook]   "Mixture of experts (MoE)" (anrans ai-infra-handbooks),
 *               "Structure" (router d->E, top-k, SwiGLU experts, weighted sum,
 *               shared expert), "Implementation: token by token vs. grouped by
 *               expert" (the naive per-token form; the stable sort by expert,
 *               per-expert counts and running start), "Load balancing"
 *               (E * sum f_i P_i, bias used only for selection).
 *  [DeepDive]   "MoE (Mixture of Experts) Deep Dive: Principles, Formulas, and
 *               Implementation", "Weighted Sum Output" (normalise the selected
 *               probabilities), "Load Balancing Loss Derivation" (N sum F_i P_i).
 *  [OneDeep]    "One Deep Concept #04 -- Mixture of Experts", section 4 "Core
 *               Innovation -- Routing" (un-renormalised y = sum_{i in T} p_i E_i).
 *
 * Parity status of each function is stated beside it; the pins live in the
 * test suite (tests/test_oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2

/* Exact widening of a stored element to double.  bf16 is the top half of an
 * IEEE binary32, so shifting its 16 bits up gives the same value exactly.
 * ORACLE_F64 inputs (e.g. dequantised FP8 weights) are used as they are. */
static double elem(const void *base, int dtype, size_t i) {
    if (dtype == ORACLE_F32) return (double)((const float *)base)[i];
    if (dtype == ORACLE_F64) return ((const double *)base)[i];
    uint32_t u = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Router for every token t:
 *   l   = W_g x_t (+ logit_bias)          [MoE-Notes] g(x) = softmax(W_g x), W_g in R^{E x d}
 *   p   = softmax(l)                      [MoE-Arch] Gating Function; [OneDeep] s4
 *   s   = l + select_bias                 [Handbook] Load balancing: the bias enters only
 *                                         the choice of the top-k, never the weights
 *   ids = the k largest s, descending,    [Handbook] Structure step 2; ties go to the lower
 *         ties to the lower expert index  expert index (the pages are silent on ties)
 *   g_j = p[ids_j], divided by sum_j g_j  [DeepDive] Weighted Sum Output (0.55, 0.3 -> /0.85);
 *         when renormalize != 0           [Handbook] route(): weights / weights.sum
 * W_g is stored [E][d] (one row of d weights per expert).
 * Outputs: topk_ids [T][k], gates [T][k], probs [T][E] (nullable), and
 * margin [T] = s_(k) - s_(k+1) (the gap between the k-th and (k+1)-th
 * selection score; +inf when k == E), nullable.
 * Pinned: worked examples, brute-force top-k, softmax special cases.
 */
int oracle_route(int T, int d, int E, int k, int dtype, const void *x, const void *w_gate,
                 const float *logit_bias, const float *select_bias, int renormalize,
                 int32_t *topk_ids, double *gates, double *probs, double *margin) {
    if (T < 0 || d < 1 || E < 1 || k < 1 || k > E) return -1;
    int bad = 0;
#pragma omp parallel
    {
        double *l = (double *)malloc(sizeof(double) * (size_t)E);
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
        double *s = (double *)malloc(sizeof(double) * (size_t)E);
        char *taken = (char *)malloc((size_t)E);
        int ok = l && p && s && taken;
        /* every thread reaches the work-sharing loop, so a failed malloc
         * cannot leave the others waiting at its barrier */
#pragma omp for schedule(static)
        for (int t = 0; t < T; ++t) {
            if (!ok) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            for (int e = 0; e < E; ++e) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i)
                    acc += elem(w_gate, dtype, (size_t)e * d + i) * elem(x, dtype, (size_t)t * d + i);
                l[e] = acc + (logit_bias ? (double)logit_bias[e] : 0.0);
            }
            double m = l[0];
            for (int e = 1; e < E; ++e)
                if (l[e] > m) m = l[e];
            double z = 0.0;
            for (int e = 0; e < E; ++e) {
                p[e] = exp(l[e] - m);
                z += p[e];
            }
            for (int e = 0; e < E; ++e) p[e] /= z;
            for (int e = 0; e < E; ++e) {
                s[e] = l[e] + (select_bias ? (double)select_bias[e] : 0.0);
                taken[e] = 0;
            }
            /* k passes of "largest remaining score, lowest index on ties". */
            double gsum = 0.0, kth = 0.0;
            for (int j = 0; j < k; ++j) {
                int best = -1;
                for (int e = 0; e < E; ++e)
                    if (!taken[e] && (best < 0 || s[e] > s[best])) best = e;
                taken[best] = 1;
                topk_ids[(size_t)t * k + j] = best;
                gates[(size_t)t * k + j] = p[best];
                gsum += p[best];
                kth = s[best];
            }
            if (renormalize)
                for (int j = 0; j < k; ++j) gates[(size_t)t * k + j] /= gsum;
            if (margin) {
                if (k == E) {
                    margin[t] = INFINITY;
                } else {
                    int nxt = -1;
                    for (int e = 0; e < E; ++e)
                        if (!taken[e] && (nxt < 0 || s[e] > s[nxt])) nxt = e;
                    margin[t] = kth - s[nxt];
                }
            }
            if (probs)
                for (int e = 0; e < E; ++e) probs[(size_t)t * E + e] = p[e];
        }
        free(l);
        free(p);
        free(s);
        free(taken);
    }
    return bad ? -2 : 0;
}

/*
 * Gates for a given set of ids: g_j = p[t, ids_j], renormalised over the k
 * chosen when renormalize != 0.  Same rule as oracle_route; used when the ids
 * come from elsewhere (a near-tie token the other side resolved differently).
 */
int oracle_gates_for_ids(int T, int E, int k, const double *probs, const int32_t *ids,
                         int renormalize, double *gates) {
    for (int t = 0; t < T; ++t) {
        double gsum = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            if (e < 0 || e >= E) return -1;
            gates[(size_t)t * k + j] = probs[(size_t)t * E + e];
            gsum += gates[(size_t)t * k + j];
        }
        if (renormalize)
            for (int j = 0; j < k; ++j) gates[(size_t)t * k + j] /= gsum;
    }
    return 0;
}

/*
 * Grouping by expert.  [Handbook] "Implementation": flatten the (token, slot)
 * pairs in the order t*k + j, sort them by expert with a STABLE sort, count
 * each expert's entries and give each expert a running start (the prefix sum
 * of the counts).  A stable sort keeps entries of one expert in flat order, so
 * an entry's rank inside its expert is the number of earlier entries (in flat
 * order) with the same expert -- which is what the single forward pass below
 * counts.
 * Capacity ([MoE-Notes] capacity and dropping; [MoE-Arch] "Tokens routed to a
 * full expert are dropped"): capacity < 0 means unlimited; otherwise an entry
 * whose rank is >= capacity is dropped.  Dropped entries get no position.
 * Outputs:
 *   counts[e]  entries routed to e (before the capacity cut)
 *   kept[e]    min(counts[e], capacity)
 *   offsets[E+1] exclusive running sum of kept
 *   rank[t*k+j]  rank inside its expert
 *   slot_pos[t*k+j] offsets[e] + rank when kept, else -1
 *   sorted_token_ids[pos] = t for every kept entry; positions past offsets[E]
 *                   are set to -1
 *   n_dropped  sum(counts) - sum(kept)
 * Pinned: brute force over tiny inputs, count/offset invariants, naive == grouped.
 */
int oracle_group(int T, int E, int k, int capacity, const int32_t *ids, int32_t *counts,
                 int32_t *kept, int32_t *offsets, int32_t *rank, int32_t *slot_pos,
                 int32_t *sorted_token_ids, int32_t *n_dropped) {
    size_t n = (size_t)T * (size_t)k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (size_t i = 0; i < n; ++i) {
        int e = ids[i];
        if (e < 0 || e >= E) return -1;
        rank[i] = counts[e];
        counts[e] += 1;
    }
    int32_t total = 0;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        kept[e] = (capacity >= 0 && counts[e] > capacity) ? capacity : counts[e];
        total += kept[e];
        offsets[e + 1] = offsets[e] + kept[e];
    }
    *n_dropped = (int32_t)n - total;
    for (size_t i = 0; i < n; ++i) sorted_token_ids[i] = -1;
    for (size_t i = 0; i < n; ++i) {
        int e = ids[i];
        if (capacity >= 0 && rank[i] >= capacity) {
            slot_pos[i] = -1;
        } else {
            int32_t pos = offsets[e] + rank[i];
            slot_pos[i] = pos;
            sorted_token_ids[pos] = (int32_t)(i / (size_t)k);
        }
    }
    return 0;
}

/*
 * One SwiGLU expert on one token, [Handbook] Structure / Expert.forward and
 * [MoE-Arch] "Each expert is a standard SwiGLU FFN":
 *   out = W2 ( silu(W1 x) (.) W3 x ),  silu(z) = z / (1 + e^{-z})
 * W1 (gate_proj) and W3 (up_proj) are stored [F][d], W2 (down_proj) [d][F]
 * (the nn.Linear [out][in] layout), each at element offset `base`.
 * h is a caller-provided scratch row of F doubles.
 */
static void swiglu_expert(int d, int F, int dtype, const void *w1, const void *w3, const void *w2,
                          size_t base1, size_t base2, const double *xt, double *h, double *out) {
    for (int f = 0; f < F; ++f) {
        double a = 0.0, b = 0.0;
        for (int i = 0; i < d; ++i) {
            a += elem(w1, dtype, base1 + (size_t)f * d + i) * xt[i];
            b += elem(w3, dtype, base1 + (size_t)f * d + i) * xt[i];
        }
        h[f] = a / (1.0 + exp(-a)) * b;
    }
    for (int o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int f = 0; f < F; ++f) acc += elem(w2, dtype, base2 + (size_t)o * F + f) * h[f];
        out[o] = acc;
    }
}

/*
 * Layer output for the tokens listed in `tokens` (n_tok of them), in the naive
 * per-token form of [Handbook] "Implementation" (outer loop over tokens, inner
 * over the k chosen experts) and [DeepDive] Code Implementation Essentials 3+5:
 *   y_t = sum_{j : slot_pos[t,j] >= 0} g_{t,j} Expert_{ids[t,j]}(x_t)
 *         + sum over shared experts of Shared(x_t)          ([MoE-Arch] s3)
 * A dropped entry (slot_pos < 0) contributes nothing ([MoE-Arch] "they
 * contribute nothing to the forward pass"); the other gates are not
 * renormalised again.  slot_pos may be NULL (nothing dropped).
 * Expert e's W1/W3 start at element e*F*d, its W2 at e*d*F.  The shared
 * expert (n_shared 0 or 1) has its own hidden size F_s.
 * y is [n_tok][d].
 */
int oracle_layer_tokens(int T, int d, int E, int k, int F, int n_shared, int F_s, int dtype,
                        const void *x, const void *w1, const void *w3, const void *w2,
                        const void *ws1, const void *ws3, const void *ws2, const int32_t *ids,
                        const double *gates, const int32_t *slot_pos, const int32_t *tokens,
                        int n_tok, double *y) {
    if (n_shared < 0 || n_shared > 1) return -1;
    int bad = 0;
    int Fmax = F > F_s ? F : F_s;
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)d);
        double *h = (double *)malloc(sizeof(double) * (size_t)(Fmax > 0 ? Fmax : 1));
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        int ok = xt && h && o;
#pragma omp for schedule(dynamic, 1)
        for (int n = 0; n < n_tok; ++n) {
            int t = tokens ? tokens[n] : n;
            double *yt = y + (size_t)n * d;
            if (!ok || t < 0 || t >= T) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            for (int i = 0; i < d; ++i) {
                xt[i] = elem(x, dtype, (size_t)t * d + i);
                yt[i] = 0.0;
            }
            for (int j = 0; j < k; ++j) {
                size_t fi = (size_t)t * k + j;
                if (slot_pos && slot_pos[fi] < 0) continue;
                int e = ids[fi];
                if (e < 0 || e >= E) continue;
                swiglu_expert(d, F, dtype, w1, w3, w2, (size_t)e * F * d, (size_t)e * d * F, xt, h, o);
                for (int i = 0; i < d; ++i) yt[i] += gates[fi] * o[i];
            }
            if (n_shared == 1) {
                swiglu_expert(d, F_s, dtype, ws1, ws3, ws2, 0, 0, xt, h, o);
                for (int i = 0; i < d; ++i) yt[i] += o[i];
            }
        }
        free(xt);
        free(h);
        free(o);
    }
    return bad ? -2 : 0;
}

/*
 * Load statistics.  [MoE-Arch] Load Balancing: L = alpha * E * sum_i f_i p_i,
 * f_i the fraction of routing decisions sent to expert i, p_i the mean router
 * probability of expert i.  [Handbook] Load balancing / aux_loss: f is the
 * per-expert count over the number of (token, slot) decisions T*k, P is the
 * mean over tokens of the softmax row.  f counts decisions before any capacity
 * cut.  probs is [T][E] (the unbiased softmax, logit_bias included).
 * Pinned: closed forms (uniform p or uniform f give alpha; the handbook's
 * skewed example gives 4 with alpha = 1), random router near 1.
 * oracle_load_stats_n takes the number of decisions n explicitly (f = counts
 * / n); expert-choice routing makes E*C decisions instead of T*k.
 */
int oracle_load_stats_n(int T, int E, long long n_decisions, const int32_t *counts, const double *probs,
                        double alpha, double *f, double *p, double *L) {
    double acc = 0.0;
    for (int e = 0; e < E; ++e) {
        f[e] = (double)counts[e] / (double)n_decisions;
        double s = 0.0;
        for (int t = 0; t < T; ++t) s += probs[(size_t)t * E + e];
        p[e] = s / (double)T;
        acc += f[e] * p[e];
    }
    *L = alpha * (double)E * acc;
    return 0;
}

/* The token-choice form: T*k decisions. */
int oracle_load_stats(int T, int E, int k, const int32_t *counts, const double *probs, double alpha, double *f,
                      double *p, double *L) {
    return oracle_load_stats_n(T, E, (long long)T * k, counts, probs, alpha, f, p, L);
}

/*
 * Auxiliary-loss-free balancing: the selection-only per-expert bias moves
 * against the load.  [MoE-Arch] s2 Load Balancing ("Over-loaded experts get a
 * negative bias"); [Handbook] Load balancing ("the bias of an overloaded
 * expert is lowered and that of an idle one raised").  The pages give the
 * direction but no step size: gamma is a parameter.
 *   load_e = counts_e (routing decisions, before any capacity cut)
 *   mean   = T k / E
 *   b_e   <- b_e - gamma * sign(load_e - mean)       (sign(0) = 0)
 * The comparison with the mean is done exactly in integers (load_e E vs T k).
 * bias_out is the exact double b_e -/+ gamma.
 * Pinned: closed forms on hand-made loads (tests/golden/bias_update_direction.txt).
 */
int oracle_bias_update(int T, int E, int k, const int32_t *counts, double gamma, const float *bias_in,
                       double *bias_out) {
    const long long total = (long long)T * (long long)k;
    for (int e = 0; e < E; ++e) {
        const long long scaled = (long long)counts[e] * (long long)E;
        const double sgn = scaled > total ? 1.0 : (scaled < total ? -1.0 : 0.0);
        bias_out[e] = (double)bias_in[e] - gamma * sgn;
    }
    return 0;
}

/*
 * Expert-choice routing ("One Deep Concept #04", section 11 "Expert Choice --
 * Reverse Who Selects Whom"): instead of each token choosing its experts, each
 * expert chooses its tokens, and every expert's bucket has the same fixed size
 * C, so the load is balanced by construction while a token may end up with any
 * number of experts (none included).  The page gives the idea, not the
 * formulas; the reading taken here:
 *   scores  p[t][e] = softmax over experts of the router logits (the same p as
 *           token choice, logit_bias included);
 *   expert e keeps the C tokens with the largest p[t][e], ties to the lower
 *           token index, listed in ascending token order;
 *   gate of (t, e) = p[t][e] (no renormalisation: a token's gates need not sum
 *           to one).
 * Selection is a library sort on (score descending, token ascending) per
 * expert -- a total order, so the chosen set is unique -- followed by a sort of
 * the C chosen token indices.
 * Outputs: sel[e*C + i] (i-th chosen token of expert e, ascending) and
 * margin[e] = p_(C) - p_(C+1), the gap between the C-th and (C+1)-th largest
 * score of expert e (+inf when C == T).  Requires 0 <= C <= T.
 * Pinned: brute force over all C-subsets on tiny tie-heavy inputs, a hand
 * example, the C = T dense limit, the closed-form balance loss.
 */
struct ec_key {
    double p;
    int t;
};

static int ec_key_cmp(const void *a, const void *b) {
    const struct ec_key *x = (const struct ec_key *)a, *y = (const struct ec_key *)b;
    if (x->p > y->p) return -1;
    if (x->p < y->p) return 1;
    return (x->t > y->t) - (x->t < y->t);
}

static int int_cmp(const void *a, const void *b) {
    const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

int oracle_ec_select(int T, int E, int C, const double *probs, int32_t *sel, double *margin) {
    if (T < 0 || E < 1 || C < 0 || C > T) return -1;
    int bad = 0;
#pragma omp parallel
    {
        struct ec_key *keys = (struct ec_key *)malloc(sizeof(struct ec_key) * (size_t)(T > 0 ? T : 1));
#pragma omp for schedule(static)
        for (int e = 0; e < E; ++e) {
            if (!keys) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            for (int t = 0; t < T; ++t) {
                keys[t].p = probs[(size_t)t * E + e];
                keys[t].t = t;
            }
            qsort(keys, (size_t)T, sizeof(struct ec_key), ec_key_cmp);
            for (int i = 0; i < C; ++i) sel[(size_t)e * C + i] = keys[i].t;
            qsort(sel + (size_t)e * C, (size_t)C, sizeof(int32_t), int_cmp);
            if (margin) margin[e] = (C == T || C == 0) ? INFINITY : keys[C - 1].p - keys[C].p;
        }
        free(keys);
    }
    return bad ? -2 : 0;
}

/*
 * Token-side view of an expert-choice assignment, in the [T][E] slot form the
 * per-token layer loop takes: slot (t, e) is live iff expert e chose token t;
 * then ids[t][e] = e, gates[t][e] = p[t][e] and slot_pos[t][e] = e*C + i, the
 * row of X_perm it occupies (expert segments of C rows, in expert order).
 * Dead slots get gates 0 and slot_pos -1.  n_empty = tokens no expert chose.
 */
int oracle_ec_slots(int T, int E, int C, const int32_t *sel, const double *probs, int32_t *ids, double *gates,
                    int32_t *slot_pos, int32_t *n_empty) {
    for (size_t i = 0; i < (size_t)T * E; ++i) {
        ids[i] = (int32_t)(i % (size_t)E);
        gates[i] = 0.0;
        slot_pos[i] = -1;
    }
    for (int e = 0; e < E; ++e)
        for (int i = 0; i < C; ++i) {
            const int t = sel[(size_t)e * C + i];
            if (t < 0 || t >= T) return -1;
            gates[(size_t)t * E + e] = probs[(size_t)t * E + e];
            slot_pos[(size_t)t * E + e] = e * C + i;
        }
    int empty = 0;
    for (int t = 0; t < T; ++t) {
        int any = 0;
        for (int e = 0; e < E; ++e) any |= slot_pos[(size_t)t * E + e] >= 0;
        empty += !any;
    }
    *n_empty = empty;
    return 0;
}


/*
 * FP8 expert weights.  The pages name FP8 (and INT4) quantisation as the way
 * to fit every expert in memory ("Mixture of Experts" notes, serving: "INT4/FP8
 * quantization is especially valuable here"; handbook, deployment: DeepSeek-V3's
 * FP8 weights) and warn that experts calibrate unevenly ("One Deep Concept
 * #04" s13), but give no format or scaling scheme.  The reading taken here:
 * OCP FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite 448; subnormals m/8 * 2^-6)
 * with one fp32 scale per output channel (per row of every weight matrix), so
 * each expert -- and each channel -- gets its own range:
 *   scale = max_i |w_i| / 448    (fp32; 1 for an all-zero row)
 *   q_i   = E4M3(w_i / scale)    (fp32 quotient, round to nearest even,
 *                                 saturating to +-448)
 *   w~_i  = value(q_i) * scale   (the weight the layer then uses; exact in fp64)
 * The quotient and the rounding are taken in fp32, as the GPU takes them, so
 * both sides choose the same code.
 * Pinned: every code's value and the rounding of random, tie and boundary
 * inputs against PyTorch's float8_e4m3fn cast; the per-row maximum maps to 448;
 * the error bound of round-to-nearest.
 */
static double e4m3_value(uint8_t c) {
    const int e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return (c & 0x80) ? -v : v;
}

static uint8_t e4m3_encode(float f) {
    if (isnan(f)) return 0x7F;
    const uint8_t sign = signbit(f) ? 0x80 : 0;
    const double a = fabs((double)f);
    if (a >= 448.0) return sign | 0x7E;  /* saturate (ties at 464 also round to 448) */
    if (a < ldexp(1.0, -6)) {           /* subnormal grid: multiples of 2^-9 */
        const double k = nearbyint(a * 512.0);   /* exact scaling; ties to even */
        return sign | (uint8_t)k;               /* k == 8 is 2^-6, code 0x08 */
    }
    int e;
    const double fr = frexp(a, &e);   /* a = fr * 2^e, fr in [0.5, 1) */
    const int E = e - 1;              /* a = (2 fr) * 2^E, 2 fr in [1, 2) */
    double k = nearbyint((2.0 * fr - 1.0) * 8.0);  /* 3-bit mantissa, ties to even */
    int Eb = E + 7;
    if (k == 8.0) {
        k = 0.0;
        Eb += 1;
    }
    if (Eb > 15 || (Eb == 15 && k == 7.0)) return sign | 0x7E;
    return sign | (uint8_t)((Eb << 3) | (int)k);
}

int oracle_e4m3_encode(int n, const float *in, uint8_t *out) {
    for (int i = 0; i < n; ++i) out[i] = e4m3_encode(in[i]);
    return 0;
}

int oracle_e4m3_decode(int n, const uint8_t *in, double *out) {
    for (int i = 0; i < n; ++i) out[i] = e4m3_value(in[i]);
    return 0;
}

int oracle_quantize_fp8(long long rows, int cols, int dtype, const void *w, uint8_t *q, float *scale) {
    if (rows < 0 || cols < 1 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16)) return -1;
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int i = 0; i < cols; ++i) {
            const float v = (float)fabs(elem(w, dtype, (size_t)r * cols + i));
            if (v > amax) amax = v;
        }
        volatile float sc = amax > 0.0f ? amax / 448.0f : 1.0f;  /* fp32 quotient */
        scale[r] = sc;
        for (int i = 0; i < cols; ++i) {
            volatile float quot = (float)elem(w, dtype, (size_t)r * cols + i) / sc;  /* fp32 quotient */
            q[(size_t)r * cols + i] = e4m3_encode(quot);
        }
    }
    return 0;
}

int oracle_dequant_fp8(long long rows, int cols, const uint8_t *q, const float *scale, double *out) {
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < rows; ++r)
        for (int i = 0; i < cols; ++i)
            out[(size_t)r * cols + i] = e4m3_value(q[(size_t)r * cols + i]) * (double)scale[r];
    return 0;
}

/*
 * Backward pass of the layer (training; the pages' own statement of the
 * gradients is the load-balancing one): for the scalar
 *   Loss = <dy, y> + dL * L_balance,
 * with the routing decisions (ids, the capacity cut) held fixed -- top-k
 * selection has no gradient ("MoE Deep Dive", Load Balancing Loss
 * Derivation: hard selection is non-differentiable) -- and f_i treated as a
 * constant while p_i carries the gradient (same section: F_i "treated as
 * constant, no gradient during backprop", P_i differentiable), the gradients
 * of every input of the forward pass, by the chain rule written out per token:
 *   kept slot j of token t, expert e, gate g:
 *     a = W1_e x, b = W3_e x, h = silu(a) b, o = W2_e h        (the expert again)
 *     dg_j  = <dy_t, o>
 *     dh    = g W2_e^T dy_t
 *     da    = dh * b * silu'(a),  silu'(a) = s (1 + a (1 - s)), s = 1/(1+e^-a)
 *     db    = dh * silu(a)
 *     dx_t += W1_e^T da + W3_e^T db
 *     dW1_e += da x^T,  dW3_e += db x^T,  dW2_e += g dy_t h^T
 *   shared expert: the same with g = 1 (no gate gradient);
 *   gates -> logits: with renormalisation the gates are the softmax of the
 *     chosen logits, dl_{e_j} = g_j (dg_j - sum_j' g_j' dg_j'), other
 *     experts 0; without it g_j = p_{e_j} and dl = p (u - <p, u>), u_{e_j} =
 *     dg_j (dropped slots have dg_j = 0);
 *   L_balance = alpha E sum_i f_i (1/T) sum_t p_ti adds
 *     dl_t += dL (alpha E / T) p_t (f - <p_t, f>),  f_i = counts_i / (T k);
 *   router: dW_g = sum_t dl_t x_t^T, dx_t += W_g^T dl_t.
 * dy is fp64 [T][d]; every output is fp64 (dx [T][d], dw_gate [E][d],
 * dw1/dw3 [E][F][d], dw2 [E][d][F], dws1/dws3 [F_s][d], dws2 [d][F_s] when
 * n_shared, dlogits [T][E]).  slot_pos < 0 marks a dropped slot.
 * Optional magnitude sums (nullable, same shapes as dw1/dw3/dw2 and the
 * shared expert's): sw1 = sum |da| |x|^T, sw3 = sum |db| |x|^T and
 * sw2 = sum |g dy| |h|^T over the same terms as the gradient entries -- the
 * scale against which a gradient computed from rounded operands is judged
 * entry by entry (rounding each factor perturbs every term in proportion
 * to its own magnitude, so the error of an entry is bounded by a multiple
 * of its magnitude sum, not of the entry itself).
 * Pinned: PyTorch autograd in fp64 on the same function; central finite
 * differences of the forward oracle; the magnitude sums equal |gradient|
 * for a single term and bound it (triangle inequality) otherwise.
 */
static double sigmoid(double a) { return 1.0 / (1.0 + exp(-a)); }

int oracle_layer_backward(int T, int d, int E, int k, int F, int n_shared, int F_s, int dtype, const void *x,
                          const void *w_gate, const float *logit_bias, const void *w1, const void *w3,
                          const void *w2, const void *ws1, const void *ws3, const void *ws2, const int32_t *ids,
                          const int32_t *slot_pos, int renormalize, double alpha, const double *dy, double dL,
                          double *dx, double *dw_gate, double *dw1, double *dw3, double *dw2, double *dws1,
                          double *dws3, double *dws2, double *dlogits, double *sw1, double *sw3, double *sw2,
                          double *sws1, double *sws3, double *sws2) {
    if (T < 1 || E < 1 || k < 1 || k > E || n_shared < 0 || n_shared > 1) return -1;
    double *gates = (double *)malloc(sizeof(double) * (size_t)T * k);
    double *fcount = (double *)calloc((size_t)E, sizeof(double));
    if (!gates || !fcount) {
        free(gates);
        free(fcount);
        return -2;
    }
    for (size_t i = 0; i < (size_t)T * k; ++i) {
        const int e = ids[i];
        if (e < 0 || e >= E) {
            free(gates);
            free(fcount);
            return -1;
        }
        fcount[e] += 1.0 / ((double)T * (double)k);
    }
    int bad = 0;
    const int Fm = F > F_s ? F : F_s;
    /* phase A, per token: gates, gate gradients, dx, dlogits */
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)d);
        double *l = (double *)malloc(sizeof(double) * (size_t)E);
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
        double *a = (double *)malloc(sizeof(double) * (size_t)Fm);
        double *b = (double *)malloc(sizeof(double) * (size_t)Fm);
        double *dh = (double *)malloc(sizeof(double) * (size_t)Fm);
        double *dg = (double *)malloc(sizeof(double) * (size_t)k);
        int ok = xt && l && p && a && b && dh && dg;
#pragma omp for schedule(dynamic, 1)
        for (int t = 0; t < T; ++t) {
            if (!ok) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const double *dyt = dy + (size_t)t * d;
            double *dxt = dx + (size_t)t * d;
            for (int i = 0; i < d; ++i) {
                xt[i] = elem(x, dtype, (size_t)t * d + i);
                dxt[i] = 0.0;
            }
            for (int e = 0; e < E; ++e) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += elem(w_gate, dtype, (size_t)e * d + i) * xt[i];
                l[e] = acc + (logit_bias ? (double)logit_bias[e] : 0.0);
            }
            double m = l[0], z = 0.0;
            for (int e = 1; e < E; ++e)
                if (l[e] > m) m = l[e];
            for (int e = 0; e < E; ++e) z += (p[e] = exp(l[e] - m));
            for (int e = 0; e < E; ++e) p[e] /= z;
            double gsum = 0.0;
            for (int j = 0; j < k; ++j) gsum += p[ids[(size_t)t * k + j]];
            for (int j = 0; j < k; ++j) {
                const double pj = p[ids[(size_t)t * k + j]];
                gates[(size_t)t * k + j] = renormalize ? pj / gsum : pj;
            }
            /* routed experts */
            for (int j = 0; j < k; ++j) {
                dg[j] = 0.0;
                if (slot_pos && slot_pos[(size_t)t * k + j] < 0) continue;
                const int e = ids[(size_t)t * k + j];
                const double g = gates[(size_t)t * k + j];
                const size_t b1 = (size_t)e * F * d, b2 = (size_t)e * d * F;
                for (int f = 0; f < F; ++f) {
                    double av = 0.0, bv = 0.0;
                    for (int i = 0; i < d; ++i) {
                        av += elem(w1, dtype, b1 + (size_t)f * d + i) * xt[i];
                        bv += elem(w3, dtype, b1 + (size_t)f * d + i) * xt[i];
                    }
                    a[f] = av;
                    b[f] = bv;
                }
                double dgj = 0.0;
                for (int o = 0; o < d; ++o) {
                    double ov = 0.0;
                    for (int f = 0; f < F; ++f) ov += elem(w2, dtype, b2 + (size_t)o * F + f) * (a[f] * sigmoid(a[f]) * b[f]);
                    dgj += dyt[o] * ov;
                }
                dg[j] = dgj;
                for (int f = 0; f < F; ++f) {
                    double acc = 0.0;
                    for (int o = 0; o < d; ++o) acc += elem(w2, dtype, b2 + (size_t)o * F + f) * dyt[o];
                    dh[f] = g * acc;
                }
                for (int f = 0; f < F; ++f) {
                    const double s = sigmoid(a[f]);
                    const double da = dh[f] * b[f] * s * (1.0 + a[f] * (1.0 - s));
                    const double db = dh[f] * a[f] * s;
                    for (int i = 0; i < d; ++i)
                        dxt[i] += elem(w1, dtype, b1 + (size_t)f * d + i) * da + elem(w3, dtype, b1 + (size_t)f * d + i) * db;
                }
            }
            /* shared expert */
            if (n_shared == 1) {
                for (int f = 0; f < F_s; ++f) {
                    double av = 0.0, bv = 0.0, acc = 0.0;
                    for (int i = 0; i < d; ++i) {
                        av += elem(ws1, dtype, (size_t)f * d + i) * xt[i];
                        bv += elem(ws3, dtype, (size_t)f * d + i) * xt[i];
                    }
                    for (int o = 0; o < d; ++o) acc += elem(ws2, dtype, (size_t)o * F_s + f) * dyt[o];
                    const double s = sigmoid(av);
                    const double da = acc * bv * s * (1.0 + av * (1.0 - s));
                    const double db = acc * av * s;
                    for (int i = 0; i < d; ++i)
                        dxt[i] += elem(ws1, dtype, (size_t)f * d + i) * da + elem(ws3, dtype, (size_t)f * d + i) * db;
                }
            }
            /* gates -> logits, plus the balance loss */
            double *dl = dlogits + (size_t)t * E;
            for (int e = 0; e < E; ++e) dl[e] = 0.0;
            if (renormalize) {
                double s = 0.0;
                for (int j = 0; j < k; ++j) s += gates[(size_t)t * k + j] * dg[j];
                for (int j = 0; j < k; ++j) dl[ids[(size_t)t * k + j]] += gates[(size_t)t * k + j] * (dg[j] - s);
            } else {
                double s = 0.0;
                for (int j = 0; j < k; ++j) s += p[ids[(size_t)t * k + j]] * dg[j];
                for (int e = 0; e < E; ++e) dl[e] -= p[e] * s;
                for (int j = 0; j < k; ++j) dl[ids[(size_t)t * k + j]] += p[ids[(size_t)t * k + j]] * dg[j];
            }
            double pf = 0.0;
            for (int e = 0; e < E; ++e) pf += p[e] * fcount[e];
            for (int e = 0; e < E; ++e) dl[e] += dL * alpha * (double)E / (double)T * p[e] * (fcount[e] - pf);
            for (int i = 0; i < d; ++i) {
                double acc = 0.0;
                for (int e = 0; e < E; ++e) acc += elem(w_gate, dtype, (size_t)e * d + i) * dl[e];
                dxt[i] += acc;
            }
        }
        free(xt);
        free(l);
        free(p);
        free(a);
        free(b);
        free(dh);
        free(dg);
    }
    if (bad) {
        free(gates);
        free(fcount);
        return -2;
    }
    /* phase B, per expert: weight gradients (each expert's rows belong to one thread) */
#pragma omp parallel
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)d);
        double *a = (double *)malloc(sizeof(double) * (size_t)Fm);
        double *b = (double *)malloc(sizeof(double) * (size_t)Fm);
        double *dh = (double *)malloc(sizeof(double) * (size_t)Fm);
        int ok = xt && a && b && dh;
#pragma omp for schedule(dynamic, 1)
        for (int e = 0; e < E + n_shared; ++e) {
            if (!ok) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const int shared = e == E;
            const int Fe = shared ? F_s : F;
            const void *W1 = shared ? ws1 : w1, *W3 = shared ? ws3 : w3, *W2 = shared ? ws2 : w2;
            const size_t b1 = shared ? 0 : (size_t)e * F * d, b2 = shared ? 0 : (size_t)e * d * F;
            double *D1 = shared ? dws1 : dw1 + b1, *D3 = shared ? dws3 : dw3 + b1, *D2 = shared ? dws2 : dw2 + b2;
            memset(D1, 0, sizeof(double) * (size_t)Fe * d);
            memset(D3, 0, sizeof(double) * (size_t)Fe * d);
            memset(D2, 0, sizeof(double) * (size_t)d * Fe);
            double *S1 = shared ? sws1 : (sw1 ? sw1 + b1 : NULL);
            double *S3 = shared ? sws3 : (sw3 ? sw3 + b1 : NULL);
            double *S2 = shared ? sws2 : (sw2 ? sw2 + b2 : NULL);
            if (S1) memset(S1, 0, sizeof(double) * (size_t)Fe * d);
            if (S3) memset(S3, 0, sizeof(double) * (size_t)Fe * d);
            if (S2) memset(S2, 0, sizeof(double) * (size_t)d * Fe);
            for (int t = 0; t < T; ++t)
                for (int j = 0; j < (shared ? 1 : k); ++j) {
                    double g = 1.0;
                    if (!shared) {
                        if (ids[(size_t)t * k + j] != e) continue;
                        if (slot_pos && slot_pos[(size_t)t * k + j] < 0) continue;
                        g = gates[(size_t)t * k + j];
                    }
                    const double *dyt = dy + (size_t)t * d;
                    for (int i = 0; i < d; ++i) xt[i] = elem(x, dtype, (size_t)t * d + i);
                    for (int f = 0; f < Fe; ++f) {
                        double av = 0.0, bv = 0.0, acc = 0.0;
                        for (int i = 0; i < d; ++i) {
                            av += elem(W1, dtype, b1 + (size_t)f * d + i) * xt[i];
                            bv += elem(W3, dtype, b1 + (size_t)f * d + i) * xt[i];
                        }
                        for (int o = 0; o < d; ++o) acc += elem(W2, dtype, b2 + (size_t)o * Fe + f) * dyt[o];
                        a[f] = av;
                        b[f] = bv;
                        dh[f] = g * acc;
                    }
                    for (int f = 0; f < Fe; ++f) {
                        const double s = sigmoid(a[f]);
                        const double da = dh[f] * b[f] * s * (1.0 + a[f] * (1.0 - s));
                        const double db = dh[f] * a[f] * s;
                        const double hf = a[f] * s * b[f];
                        for (int i = 0; i < d; ++i) {
                            D1[(size_t)f * d + i] += da * xt[i];
                            D3[(size_t)f * d + i] += db * xt[i];
                        }
                        for (int o = 0; o < d; ++o) D2[(size_t)o * Fe + f] += g * dyt[o] * hf;
                        if (S1)
                            for (int i = 0; i < d; ++i) S1[(size_t)f * d + i] += fabs(da) * fabs(xt[i]);
                        if (S3)
                            for (int i = 0; i < d; ++i) S3[(size_t)f * d + i] += fabs(db) * fabs(xt[i]);
                        if (S2)
                            for (int o = 0; o < d; ++o) S2[(size_t)o * Fe + f] += fabs(g * dyt[o]) * fabs(hf);
                    }
                }
        }
        free(xt);
        free(a);
        free(b);
        free(dh);
    }
    /* router weight gradient */
#pragma omp parallel for schedule(static)
    for (int e = 0; e < E; ++e)
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int t = 0; t < T; ++t) acc += dlogits[(size_t)t * E + e] * elem(x, dtype, (size_t)t * d + i);
            dw_gate[(size_t)e * d + i] = acc;
        }
    free(gates);
    free(fcount);
    return bad ? -2 : 0;
}
