/*
 * moe_b300.h -- C ABI of libmoe_b300.so: the forward pass of a Mixture-of-Experts
 * SwiGLU FFN layer on one NVIDIA B300 (sm_103a).
 *
 * What the layer computes (sources by page title and section):
 *   1. router logits  l = W_g x (+ logit_bias)      "Mixture of Experts" notes, How it works
 *                                                    (g(x) = softmax(W_g x), W_g in R^{E x d});
 *                                                    "MoE Architecture" s2 Gating Function
 *   2. p = softmax(l)                                same; "One Deep Concept #04" s4
 *   3. top-k of l + select_bias, gates g_j = p[id_j] "Mixture of experts (MoE)" handbook,
 *      renormalised to sum 1 (optional)             Structure and Load balancing (bias used
 *                                                    only for the choice); "MoE Deep Dive",
 *                                                    Weighted Sum Output (divide by the sum)
 *   4. grouping by expert: counts, stable ranks,    handbook, "Implementation: token by token
 *      capacity cut, offsets, permutation           vs. grouped by expert" (stable argsort,
 *                                                    bincount, running start); notes,
 *                                                    capacity and token dropping
 *   5. per expert segment: H = silu(X W1^T) * (X W3^T), Y = H W2^T   handbook Structure
 *                                                    (Expert: down(silu(gate(x)) * up(x)));
 *                                                    "MoE Architecture" s3 (SwiGLU experts)
 *   6. y_t = sum_j g_j Y[pos(t,j)] + Shared(x_t)     handbook forward_grouped / forward_naive;
 *                                                    "MoE Architecture" s3 Shared Experts
 *   7. f_i = counts_i/(T k), p_i = mean_t p[t,i],   "MoE Architecture" s2 Load Balancing;
 *      L_balance = alpha E sum_i f_i p_i             handbook Load balancing (aux_loss)
 *
 * Expert-choice routing (cfg->routing = MOE_ROUTE_EXPERT_CHOICE; "One Deep
 * Concept #04" s11, Expert Choice -- Reverse Who Selects Whom) replaces steps
 * 3-4: every expert takes a fixed bucket of C tokens, those with the largest
 * p[t][e] (ties to the lower token index), so each expert's load is exactly C
 * and a token gets any number of experts, zero included; the gate of a chosen
 * (t, e) is p[t][e] (never renormalised).  Steps 5-7 are unchanged, with the
 * E*C chosen pairs in place of the T*k routing decisions.
 *
 * Conventions for every entry point
 *   - Every pointer argument except `cfg` and `stats` (a host struct of device
 *     pointers) is a DEVICE pointer unless stated otherwise.  The caller owns all
 *     memory; the library never allocates, frees or keeps a pointer past the call.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and the call returns without synchronising.  Results are valid
 *     once the stream has reached that point.
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_* code.  Argument errors
 *     are detected on the host before anything is enqueued.  MOE_ERR_CUDA
 *     reports a launch failure (cudaGetLastError after the launches).
 *     Failures found by a kernel (a bounded wait that ran out, an index out of
 *     range) are recorded in the workspace's status word and are read with
 *     moe_last_device_status after the stream is synchronised.
 *   - Layouts are row-major.  x is [T][d]; W_g is [E][d] (one row per expert,
 *     the notes' W_g in R^{E x d}, i.e. an nn.Linear(d, E) weight);
 *     W1 (gate_proj) and W3 (up_proj) are [E][F][d]; W2 (down_proj) is
 *     [E][d][F]; the shared expert's Ws1/Ws3 are [F_s][d] and Ws2 is [d][F_s].
 *   - dtype MOE_BF16: x, weights and y are bf16; accumulation is fp32; the
 *     hidden activation H is stored as bf16 between the two expert GEMMs (or
 *     as a hi + lo bf16 pair when cfg->h_split).
 *     dtype MOE_F32: everything is fp32 (IEEE fp32 FMA, no TF32).
 *   - Alignment: every device pointer must be 16-byte aligned and the
 *     workspace 256-byte aligned; d, F and F_s must be multiples of 8.
 *   - Limits: 1 <= k <= min(E, 32); E <= 1024; T >= 0; T * k < 2^31 (expert
 *     choice: also T * E < 2^31 and E * C < 2^31);
 *     n_shared is 0 or 1; d, F, F_s >= 8.  With T = 0 a call validates cfg
 *     only and enqueues nothing (pointers may then be NULL).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st *moe_stream_t;

enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 };

/* Who chooses whom (moe_config.routing). */
enum moe_routing { MOE_ROUTE_TOKEN_CHOICE = 0, MOE_ROUTE_EXPERT_CHOICE = 1 };

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_NULL = -1,          /* a required pointer is NULL                          */
    MOE_ERR_SHAPE = -2,         /* sizes out of range or misaligned (see Limits)       */
    MOE_ERR_DTYPE = -3,         /* unknown dtype                                       */
    MOE_ERR_WORKSPACE = -4,     /* ws_bytes < moe_workspace_size(cfg) or ws misaligned */
    MOE_ERR_CUDA = -5,          /* a kernel launch or CUDA runtime call failed         */
    MOE_ERR_DEVICE = -6,        /* current device is not a compute-capability 10.3 GPU */
    MOE_ERR_TIMEOUT = -7,       /* device: a bounded wait ran out (kernel gave up)     */
    MOE_ERR_DEVICE_BOUNDS = -8, /* device: an index read from memory was out of range  */
    MOE_ERR_ALIGN = -9          /* a device pointer is not 16-byte aligned             */
};

/* Layer description.  T tokens, model width d, E routed experts, top-k, expert
 * hidden size d_ff (F); n_shared (0 or 1) always-on shared experts of hidden
 * size d_ff_shared (F_s).  capacity < 0: no limit; otherwise each expert keeps
 * at most `capacity` (token, slot) entries, the ones with the lowest token
 * index, and drops the rest (a dropped entry contributes nothing; the other
 * gates are not renormalised again).  alpha scales L_balance. */
typedef struct moe_config {
    int32_t T, d, E, k, d_ff;
    int32_t n_shared, d_ff_shared;
    int32_t dtype;       /* enum moe_dtype                                     */
    int32_t renormalize; /* 1: divide the k gates of a token by their sum     */
    int32_t capacity;    /* < 0: unlimited                                     */
    float alpha;         /* L_balance = alpha * E * sum_i f_i p_i              */
    int32_t y_fp32;      /* 0: y in `dtype`; 1: y in fp32 (the combine's fp32
                            sum, before any rounding to bf16)                  */
    int32_t h_split;     /* bf16 layers: 1 keeps the SwiGLU activation H as a
                            pair of bf16 values (hi + lo, ~16 significant bits)
                            and runs the down GEMM on both halves, for layers
                            whose outputs are too heavy-tailed for a bf16 H;
                            costs a second pass of the down GEMM's MMAs.
                            Ignored for fp32 layers.                           */
    int32_t routing;     /* enum moe_routing.  MOE_ROUTE_EXPERT_CHOICE: each
                            expert takes a bucket of C tokens, C = capacity
                            when capacity > 0, else floor(T k / E) (k read as
                            the average number of experts per token), clamped
                            to [1, T]; renormalize and select_bias have no
                            effect (a per-expert constant does not change an
                            expert's ranking of the tokens).                   */
    int32_t yperm_bf16;  /* bf16 layers: 1 stores each expert row of the down
                            GEMM (y_perm, after its gate) and the shared
                            expert's rows (y_shared) in bf16 instead of fp32,
                            rounded once per row after its K slices are summed,
                            halving the combine's reads; the combine still adds
                            them in fp32.  For layers with many experts per
                            token, whose rows are each a small part of y.
                            0 for fp32 layers.                                 */
} moe_config;

/* Optional statistics outputs of moe_forward (device pointers, each nullable). */
typedef struct moe_stats {
    int32_t *counts;    /* [E]  routing decisions per expert, before the capacity cut */
    int32_t *kept;      /* [E]  min(counts, capacity)                                */
    float *f;           /* [E]  counts / (T k)                                       */
    float *p;           /* [E]  mean over tokens of the softmax row                  */
    float *L;           /* [1]  alpha * E * sum f p                                  */
    int32_t *n_dropped; /* [1]  T k - sum kept                                       */
} moe_stats;
/* Under expert choice: counts = kept = C for every expert, f = C / (E C) =
 * 1/E (so L = alpha * sum_e p_e = alpha), and n_dropped counts the tokens that
 * no expert took (they receive only the shared expert's output, or 0). */

/* Bytes of device workspace every entry point below may use for `cfg`.
 * Returns 0 when cfg is invalid.  The workspace needs 256-byte alignment. */
MOE_API size_t moe_workspace_size(const moe_config *cfg);

/* Prepares a freshly allocated workspace: zeroes its device status word and
 * the completion counters some kernels keep in it (enqueued on `stream`).
 * Call once per workspace before the first entry point; every kernel leaves
 * its counters at zero again, and moe_last_device_status clears the word (and,
 * after a device error, the counters) again after reading it.
 * Errors: MOE_ERR_NULL, MOE_ERR_WORKSPACE, MOE_ERR_CUDA. */
MOE_API int moe_workspace_init(const moe_config *cfg, void *ws, size_t ws_bytes, moe_stream_t stream);

/* Router, softmax and top-k (steps 1-3).
 *   x [T][d], w_gate [E][d] (dtype), logit_bias [E] fp32 or NULL (added to the
 *   logits everywhere: selection, gates and p), select_bias [E] fp32 or NULL
 *   (added to the logits for the top-k choice only).
 *   Outputs: topk_ids int32 [T][k] (descending selection score, ties to the lower
 *   expert index), gates fp32 [T][k] (unbiased softmax at those ids, renormalised
 *   when cfg->renormalize), p_mean fp32 [E] or NULL (mean softmax row).
 *   A NaN selection score ranks below every other score (as -inf), so a token
 *   with non-finite inputs still gets k distinct valid ids; its gates, and the
 *   layer's output row for it, are then NaN.  Other tokens are unaffected. */
MOE_API int moe_route(const moe_config *cfg, const void *x, const void *w_gate, const float *logit_bias,
              const float *select_bias, int32_t *topk_ids, float *gates, float *p_mean, void *ws,
              size_t ws_bytes, moe_stream_t stream);

/* Expert-choice routing and grouping in one step (requires cfg->routing ==
 * MOE_ROUTE_EXPERT_CHOICE; token-choice configurations get MOE_ERR_SHAPE, as
 * do moe_route, moe_permute, moe_permute_static and moe_bias_update under
 * expert choice).  Router logits and softmax as in moe_route (logit_bias
 * nullable), then every expert e takes its C tokens (bucket size in
 * moe_config.routing) as rows [e*C, (e+1)*C) of the permuted layout, in
 * ascending token order.
 *   Outputs: probs fp32 [T][E] (the softmax rows; nullable -- the workspace
 *   keeps a copy), sorted_token_ids int32 [E*C], gates_perm fp32 [E*C] (p of
 *   each chosen pair), slot_pos int32 [T][E] (row of pair (t, e), -1 when
 *   expert e did not take t), offsets int32 [E+1] (= e*C), p_mean fp32 [E]
 *   (nullable), x_perm [E*C][d] (dtype; nullable: row r = x[sorted_token_ids[r]]).
 * moe_expert_ffn then takes x_perm, offsets and gates_perm unchanged, and
 * moe_combine takes slot_pos as its [T][E] slot map. */
MOE_API int moe_route_expert_choice(const moe_config *cfg, const void *x, const void *w_gate,
                                    const float *logit_bias, float *probs, int32_t *sorted_token_ids,
                                    float *gates_perm, int32_t *slot_pos, int32_t *offsets, float *p_mean,
                                    void *x_perm, void *ws, size_t ws_bytes, moe_stream_t stream);

/* Grouping by expert (step 4).  Entries are the (t, j) pairs in flat order
 * t*k + j; an entry's rank is the number of earlier entries of the same expert.
 *   In:  topk_ids int32 [T][k], gates fp32 [T][k], x [T][d] (dtype).
 *   Out: counts [E], kept [E], offsets [E+1] (exclusive running sum of kept),
 *        sorted_token_ids [T*k] (token of the entry at each position; positions
 *        >= offsets[E] are set to -1), slot_pos [T][k] (position of the entry,
 *        -1 if dropped), gates_perm fp32 [T*k] (gate at each position, 0 past the
 *        end), x_perm [T*k][d] (dtype; row pos = x[sorted_token_ids[pos]];
 *        rows past offsets[E] are left untouched), n_dropped [1].
 * All outputs are required (non-NULL). */
MOE_API int moe_permute(const moe_config *cfg, const int32_t *topk_ids, const float *gates, const void *x,
                int32_t *counts, int32_t *kept, int32_t *offsets, int32_t *sorted_token_ids,
                int32_t *slot_pos, float *gates_perm, void *x_perm, int32_t *n_dropped, void *ws,
                size_t ws_bytes, moe_stream_t stream);

/* Allocation-free variant of moe_permute (the pages have no counterpart; it
 * exists for callers, not for the method).  Same arguments and outputs as
 * moe_permute, minus the workspace: for callers that are handed only their
 * input and output buffers (a plug-in slot with a fixed signature) or that
 * run where device allocation is forbidden after start-up, and so cannot
 * obtain a workspace.  The per-block histogram scratch lives instead in a
 * fixed device array inside the library: 65,536 int32 (256 KiB), held on
 * every device that loads the library until the process exits.
 *   Limit: ceil(T / 64) * E must not exceed 65,536, else MOE_ERR_SHAPE and
 *   nothing is enqueued (e.g. T = 16384 with E <= 256, T = 4096 with E <= 1024).
 *   The call allocates nothing and calls no allocating routine.  Its first
 *   call on a device looks up the array's device address (once per device,
 *   with that device current); make that first call before any stream capture.
 *   With the CUDA runtime's lazy module loading (the default), that first call
 *   is also when the library's device code, and with it the array, is loaded
 *   onto the device: a caller whose runtime forbids device allocation after
 *   start-up makes its first call on each device during start-up.
 *   All calls on a device share the one array and each call overwrites what
 *   the previous one left there, so calls whose kernels overlap on the GPU
 *   (different streams without ordering) race and give wrong results;
 *   serialise them.  There is no workspace status word: ids outside [0, E)
 *   are skipped, not reported. */
MOE_API int moe_permute_static(const moe_config *cfg, const int32_t *topk_ids, const float *gates,
                               const void *x, int32_t *counts, int32_t *kept, int32_t *offsets,
                               int32_t *sorted_token_ids, int32_t *slot_pos, float *gates_perm,
                               void *x_perm, int32_t *n_dropped, moe_stream_t stream);

/* Expert FFNs over the grouped rows (step 5), gate applied in the epilogue.
 *   x_perm [T*k][d] and offsets [E+1] as produced by moe_permute (expert
 *   choice: [E*C][d] from moe_route_expert_choice); gates_perm fp32
 *   [T*k]; w1, w3 [E][F][d], w2 [E][d][F] (dtype).
 *   y_perm [T*k][d] (fp32, or bf16 when cfg->yperm_bf16): row pos =
 *   gates_perm[pos] * W2_e(silu(W1_e x) * W3_e x) for pos < offsets[E] (rows
 *   past the end are left untouched).
 *   Shared expert (when cfg->n_shared == 1): x [T][d], ws1, ws3 [F_s][d],
 *   ws2 [d][F_s] and y_shared [T][d] (as y_perm) = Shared(x) (gate 1) are
 *   required; when n_shared == 0 those five may be NULL. */
MOE_API int moe_expert_ffn(const moe_config *cfg, const void *x_perm, const int32_t *offsets,
                   const float *gates_perm, const void *w1, const void *w3, const void *w2,
                   const void *x, const void *ws1, const void *ws3, const void *ws2, void *y_perm,
                   void *y_shared, void *ws, size_t ws_bytes, moe_stream_t stream);

/* Combine (step 6): y[t] = sum over j = 0..k-1 with slot_pos[t][j] >= 0 of
 * y_perm[slot_pos[t][j]], in that order, plus y_shared[t] when y_shared is
 * non-NULL; accumulated in fp32 and stored in cfg->dtype (round to nearest
 * even for bf16), or in fp32 when cfg->y_fp32.  y_perm and y_shared are fp32,
 * or bf16 when cfg->yperm_bf16 (as moe_expert_ffn writes them).  A token whose
 * entries were all dropped gets only its shared row (or 0).  Under expert
 * choice slot_pos is [T][E] and the sum runs over j = 0..E-1. */
MOE_API int moe_combine(const moe_config *cfg, const void *y_perm, const int32_t *slot_pos,
                const void *y_shared, void *y, moe_stream_t stream);

/* Load statistics (step 7) from counts [E] (moe_permute) and p_mean [E]
 * (moe_route): f [E] = counts/(T k), L [1] = alpha * E * sum f p_mean.
 * f or L may be NULL.  Under expert choice the denominator is E*C (the
 * number of chosen pairs) instead of T k. */
MOE_API int moe_load_stats(const moe_config *cfg, const int32_t *counts, const float *p_mean, float *f,
                   float *L, moe_stream_t stream);

/* Selection-bias update of auxiliary-loss-free balancing ("MoE Architecture"
 * s2 Load Balancing: over-loaded experts get a negative bias; "Mixture of
 * experts (MoE)" handbook, Load balancing: an overloaded expert's bias is
 * lowered and an idle one's raised).  A training-time step between layer
 * calls, not part of the forward pass:
 *   select_bias[e] -= gamma * sign(counts[e] - T k / E)      (sign(0) = 0)
 * with counts [E] int32 as produced by moe_permute / moe_forward (routing
 * decisions before the capacity cut; the comparison with the mean is exact).
 * select_bias [E] fp32 is updated in place.  The pages give no step size:
 * gamma is the caller's. */
MOE_API int moe_bias_update(const moe_config *cfg, const int32_t *counts, float gamma, float *select_bias,
                            moe_stream_t stream);

/* The whole layer (steps 1-7) in one call, fused where the steps allow.
 *   y [T][d] (dtype, or fp32 when cfg->y_fp32) receives the layer output; stats (host struct, nullable)
 *   names optional device outputs.  ws1/ws3/ws2 are the shared expert's weights
 *   (required iff cfg->n_shared == 1).
 *   Token-choice bf16 one-token batches (T = 1) with E <= 32, k <= 16 and a
 *   single bf16 H run as two kernels (moe_plan_describe: up=fused): every CTA
 *   routes the batch itself (the one-block-per-token router's arithmetic, so
 *   ids, gates and statistics are bit for bit those of moe_route), the first
 *   kernel streams W1/W3 rows and writes H, the second streams W2 rows and
 *   writes y with the gates and the shared expert applied.  The expert dots
 *   run on the CUDA cores with fp32 accumulation, so y agrees with
 *   the step-by-step entry points to rounding, not bit for bit. */
MOE_API int moe_forward(const moe_config *cfg, const void *x, const void *w_gate, const float *logit_bias,
                const float *select_bias, const void *w1, const void *w3, const void *w2,
                const void *ws1, const void *ws3, const void *ws2, void *y, const moe_stats *stats,
                void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---- FP8 expert weights ------------------------------------------------
 * The pages name FP8 quantisation of the experts as the way to fit every
 * expert in memory ("Mixture of Experts" notes, serving; handbook, DeepSeek-V3
 * in FP8) without fixing a scheme.  Here: OCP E4M3 codes (bias 7, largest
 * finite 448, no infinities) with one fp32 scale per output channel, i.e. per
 * row of every weight matrix:
 *   scale_r = max_i |w_ri| / 448 (1 for an all-zero row),
 *   q_ri    = E4M3(w_ri / scale_r)  (IEEE fp32 quotient, round to nearest
 *             even, saturating), and the layer uses w~_ri = value(q_ri) scale_r.
 * The expert GEMMs stream the one-byte codes (half the bytes of bf16 weights:
 * the decode-time bound) and apply scale_r to the fp32 accumulator of output
 * channel r.  Prefill-sized batches widen the codes exactly to bf16 in shared
 * memory (bf16 x bf16 MMAs).  Batches the two fused small-batch kernels take
 * (see moe_forward) convert the codes exactly to f16 on the CUDA cores and
 * multiply them by x and H held as f16, each warp's slice of a row scaled by
 * a power of two that puts its largest magnitude in [0.5, 1): the 16 products
 * of each 16-code vector are summed as two f16 partial sums of eight, which
 * then join an fp32 accumulator.  Other decode-sized batches (at most 32 rows per touched
 * expert on average) feed the codes to the FP8 tensor cores as they are; that MMA takes FP8 on both sides, so every bf16 row of x and of H is
 * first split into two E4M3 code rows and a power-of-two scale,
 * row = s (hi + lo), which reproduces every entry within a factor 2^10 of the
 * row's largest magnitude exactly (smaller entries: absolute error at most
 * 2^-17 times that magnitude).  Both products then accumulate in fp32. */

/* Quantises a [rows][cols] matrix (dtype MOE_BF16 or MOE_F32; cols a multiple
 * of 16) row by row: q [rows][cols] uint8 codes, scale [rows] fp32.  Device
 * pointers, 16-byte aligned.  Quantise W1 and W3 as [E*F][d] and W2 as
 * [E*d][F] (and the shared expert's matrices the same way).
 * Errors: MOE_ERR_NULL, MOE_ERR_SHAPE, MOE_ERR_DTYPE, MOE_ERR_ALIGN, MOE_ERR_CUDA. */
MOE_API int moe_quantize_fp8(const void *w, int32_t dtype, int64_t rows, int32_t cols, uint8_t *q, float *scale,
                             moe_stream_t stream);

/* FP8 weights of the routed experts (and of the shared expert when
 * cfg->n_shared == 1; those six pointers may be NULL otherwise). */
typedef struct moe_fp8_weights {
    const uint8_t *w1, *w3; /* [E][F][d] codes               */
    const uint8_t *w2;      /* [E][d][F] codes               */
    const float *s1, *s3;   /* [E][F] scales (rows of W1/W3) */
    const float *s2;        /* [E][d] scales (rows of W2)    */
    const uint8_t *ws1, *ws3, *ws2; /* shared: [F_s][d], [F_s][d], [d][F_s] codes */
    const float *ss1, *ss3, *ss2;   /* shared: [F_s], [F_s], [d] scales          */
} moe_fp8_weights;

/* moe_forward with FP8 expert weights (host struct of device pointers).
 * cfg->dtype must be MOE_BF16 (x, w_gate and y stay bf16; the router is
 * unchanged) and cfg->h_split 0; d, F and F_s must be multiples of 16.  Both
 * routings; same workspace, statistics and errors as moe_forward. */
MOE_API int moe_forward_fp8(const moe_config *cfg, const void *x, const void *w_gate, const float *logit_bias,
                            const float *select_bias, const moe_fp8_weights *w, void *y, const moe_stats *stats,
                            void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---- backward pass ------------------------------------------------------
 * Gradients of the scalar  <dy, y> + dL * L_balance  with respect to x, W_g,
 * W1, W3, W2 and the shared expert's weights, the routing decisions (top-k
 * ids and the capacity cut) held fixed -- hard selection has no gradient --
 * and f_i held constant while p_i carries the gradient ("MoE Deep Dive", Load
 * Balancing Loss Derivation: F_i is a constant statistic, P_i the
 * differentiable soft probability).  Per kept slot (expert e, gate g):
 *   dg = <dy, W2_e h>,  dh = g W2_e^T dy,  dG = dh U silu'(G),  dU = dh silu(G),
 *   dx += W1_e^T dG + W3_e^T dU,  dW1_e += dG x^T,  dW3_e += dU x^T,
 *   dW2_e += g dy h^T;  gates -> logits through the (renormalised) softmax;
 *   L_balance adds dL alpha E / T  p_t (f - <p_t, f>) to the logits of t;
 *   dW_g = sum_t dlogits_t x_t^T,  dx += W_g^T dlogits.
 * The call recomputes the forward routing, grouping and expert activations
 * (nothing is kept from moe_forward) on the tensor-core GEMMs, with bf16
 * operands (G, U, dG, dU, h and g*dy rounded to bf16 where they feed a GEMM)
 * and fp32 accumulation.
 *   In:  x [T][d], w_gate, w1, w3, w2 (and ws1, ws3, ws2 when n_shared) as for
 *        moe_forward, logit_bias / select_bias nullable, dy [T][d] (bf16),
 *        dL (host float, the upstream gradient of L_balance; 0 to ignore it).
 *   Out (fp32, caller-owned): dx [T][d], dw_gate [E][d], dw1, dw3 [E][F][d],
 *        dw2 [E][d][F]; dws1, dws3 [F_s][d], dws2 [d][F_s] when n_shared.
 * Requires cfg->dtype == MOE_BF16 (else MOE_ERR_DTYPE) and token-choice
 * routing (expert choice: MOE_ERR_SHAPE); ws of moe_backward_workspace_size
 * bytes (it covers a forward workspace as well). */
MOE_API size_t moe_backward_workspace_size(const moe_config *cfg);
MOE_API int moe_backward(const moe_config *cfg, const void *x, const void *w_gate, const float *logit_bias,
                         const float *select_bias, const void *w1, const void *w3, const void *w2, const void *ws1,
                         const void *ws3, const void *ws2, const void *dy, float dL, float *dx, float *dw_gate,
                         float *dw1, float *dw3, float *dw2, float *dws1, float *dws3, float *dws2, void *ws,
                         size_t ws_bytes, moe_stream_t stream);

/* ---- training step: forward that keeps its activations ------------------
 * moe_forward_train computes y and the statistics as moe_forward does (for
 * decode-sized batches it keeps the large-batch GEMMs, so y may differ from
 * moe_forward's in rounding), and leaves in ws -- a moe_backward_workspace_size workspace -- what the
 * backward pass would otherwise recompute: the softmax rows, the top-k ids,
 * gates and grouping, x in expert order, and the fp32 pre-activations
 * G = x W1^T, U = x W3^T of every kept slot (and of the shared expert).  The
 * up GEMM writes G and U from the same accumulators that give h = silu(G) U,
 * so moe_backward_saved on that workspace returns the gradients moe_backward
 * returns, bit for bit, without the routing, grouping and two of the seven
 * expert GEMMs (the FLOPs of the forward up GEMM).  The gradients are those
 * of "MoE Deep Dive", Load Balancing Loss Derivation (see moe_backward).
 *   moe_forward_train: arguments and outputs as moe_forward (bf16, token
 *   choice, cfg->h_split 0; else MOE_ERR_DTYPE / MOE_ERR_SHAPE), ws of
 *   moe_backward_workspace_size bytes (MOE_ERR_WORKSPACE if smaller).
 *   moe_backward_saved: arguments, outputs and errors as moe_backward; the
 *   caller passes the cfg, x, weights, biases and ws of the last
 *   moe_forward_train on that ws, with no other call on ws in between.  The
 *   library cannot check this, and not every index it reads back from ws is
 *   re-checked on the device: any other workspace content is a caller error
 *   with undefined results.  Both are asynchronous on `stream`. */
MOE_API int moe_forward_train(const moe_config *cfg, const void *x, const void *w_gate, const float *logit_bias,
                              const float *select_bias, const void *w1, const void *w3, const void *w2,
                              const void *ws1, const void *ws3, const void *ws2, void *y, const moe_stats *stats,
                              void *ws, size_t ws_bytes, moe_stream_t stream);
MOE_API int moe_backward_saved(const moe_config *cfg, const void *x, const void *w_gate, const float *logit_bias,
                               const float *select_bias, const void *w1, const void *w3, const void *w2,
                               const void *ws1, const void *ws3, const void *ws2, const void *dy, float dL,
                               float *dx, float *dw_gate, float *dw1, float *dw3, float *dw2, float *dws1,
                               float *dws3, float *dws2, void *ws, size_t ws_bytes, moe_stream_t stream);

/* Reads (and clears) the device status word kept in the workspace: MOE_OK,
 * MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_BOUNDS.  Synchronises `stream` first.
 * Returns MOE_ERR_CUDA if the copy itself fails. */
MOE_API int moe_last_device_status(const moe_config *cfg, void *ws, moe_stream_t stream);

/* ---- diagnostics ---------------------------------------------------------
 * Stage timing hook.  While set (per host thread), every entry point records
 * events[2*s] on its stream just before the launches of stage s and
 * events[2*s+1] just after them, for s = 0 router (logits, softmax, top-k),
 * 1 grouping scan (ranks, offsets, permutation; includes the histogram
 * kernel of moe_permute), 2 token rows for the up GEMM (the x_perm gather;
 * with FP8 weights on decode-sized batches, the E4M3 hi/lo split of x),
 * 3 up GEMM (SwiGLU, and its split-K finalize), 4 down GEMM (with FP8 weights
 * on decode-sized batches, after the E4M3 hi/lo split of H), 5 combine (a
 * decode-sized batch is grouped inside the router launch, so stage 1 records
 * nothing there).  `events` holds n (<= 12) cudaEvent_t handles owned by
 * the caller; NULL entries are skipped.  Pass events = NULL to clear.  On a
 * stream that is being captured into a CUDA graph the events are recorded
 * as external event nodes, so every replay of the graph records them.
 * Returns MOE_OK, or MOE_ERR_SHAPE if n is out of range. */
MOE_API int moe_set_stage_events(void *const *events, int n);

/* Number of kernels this library has launched in this process so far. */
MOE_API uint64_t moe_launch_count(void);

/* Static text for a status code (never NULL). */
MOE_API const char *moe_strerror(int status);

/* Diagnostic: the kernels moe_forward picks for this configuration, as one
 * line of "key=value" words written into buf (NUL-terminated, truncated to
 * len bytes): router=split_d|warp|gemm|fused, up=/down=
 * tc|tc_pair|tc_decode32|tc_decode64|simt|fused (tc_pair = CTA-pair
 * tensor-core GEMM with 256-row tiles; tc_decode = weights on the MMA's M side
 * with 32 or 64 token rows; fused = the two small-batch kernels, with bf16
 * weights), ksplit_up=/ksplit_down= the
 * split-K factor, gather_a=1 when the up GEMM gathers x rows itself, h= the
 * storage of the SwiGLU output.  The choice depends on the configuration
 * only, never on the data.  No counterpart on the pages.  Returns MOE_OK,
 * MOE_ERR_NULL (buf NULL or len 0) or a configuration error. */
MOE_API int moe_plan_describe(const moe_config *cfg, char *buf, size_t len);

/* Test switch for failure detection (no counterpart on the pages): with
 * on != 0, every tensor-core GEMM launched afterwards in this process (any
 * thread, any device) issues no operand loads and bounds its waits at 20 ms
 * instead of 2 s, so its consumers give up, record MOE_ERR_TIMEOUT in the
 * workspace status word, free their tensor memory and return, leaving the
 * context usable; on = 0 restores normal launches.  Nothing faults or hangs
 * either way.  Off at load.  Returns the previous setting (0 or 1). */
MOE_API int moe_test_stall_gemm(int on);

/* Library version as "major.minor.patch". */
MOE_API const char *moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
