// common.cuh -- internal declarations shared by the kernels of libmoe_b300.so.
//
// Nothing here is part of the C ABI (include/moe_b300.h is).  The launchers
// declared at the bottom are called only by api.cu, which validates every
// argument before a launch.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_b300.h"

namespace moe {

// Upper bound on E handled by the kernels (shared-memory histograms, scans).
constexpr int kMaxExperts = 1024;
// The router emits one expert histogram (and one partial sum of p) per chunk
// of consecutive tokens; the grouping scan reads those rows, chunked the same
// way.  Chunk sizes per router kernel:
constexpr int kRouterTokensPerBlock = 64;  // logits router; the stand-alone moe_permute histograms
constexpr int kWarpRouterChunk = 32;       // warp router (prefill-sized batches, small E)
constexpr int kSplitDRouterMaxT = 256;     // up to this many tokens: one block per token
constexpr int kRouterThreads = 256;
// The fused warp router keeps E logits per lane in registers and W_g in
// shared memory (padded to 8 or 16 rows); larger routers go through the
// tensor-core GEMM.
constexpr int kWarpRouterMaxE = 16;
constexpr int kWarpRouterThreads = 512;
constexpr size_t kWarpRouterMaxSmem = 160 * 1024;

inline int warp_router_width(int E) { return E <= 8 ? 8 : 16; }

inline size_t warp_router_smem_bytes(int E, int d, int dtype) {
    return (size_t)warp_router_width(E) * d * (dtype == MOE_BF16 ? 2 : 4);
}

// True when the fused warp router handles this layer.
inline bool use_warp_router(int E, int d, int dtype) {
    return E <= kWarpRouterMaxE && warp_router_smem_bytes(E, d, dtype) <= kWarpRouterMaxSmem;
}

// True when the one-block-per-token router handles this layer (decode-sized
// batches: every token gets a whole block, d split across its threads).
inline bool use_split_d_router(int T, int E) { return T <= kSplitDRouterMaxT && E <= 32; }

// Tokens per histogram row for the router a layer uses (T, E, d, dtype).
inline int router_chunk(int T, int E, int d, int dtype) {
    if (use_split_d_router(T, E)) return 1;
    if (use_warp_router(E, d, dtype)) return kWarpRouterChunk;
    return kRouterTokensPerBlock;
}

// Device status word values (mirror enum moe_status).
constexpr int kStatusTimeout = MOE_ERR_TIMEOUT;
constexpr int kStatusBounds = MOE_ERR_DEVICE_BOUNDS;

// Programmatic dependent launch.  Every kernel of this library is launched
// with launch_pdl and calls pdl_wait() before its first global-memory access.
// A dependent may rely only on what its predecessor wrote before triggering,
// so a kernel triggers (pdl_trigger) only after its CTA's last global write
// -- or not at all, which triggers at exit.  What overlaps is the successor's
// launch and its memory-free prologue (barrier set-up, TMEM allocation,
// tensor-map prefetch) with the predecessor's last CTAs.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ void record_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Column sums over the per-chunk rows of the router's statistics (p and the
// expert histograms), for layers with at most kWarpColumnMaxE experts: one
// warp per column, lane j taking rows j, j+32, ... in ascending order, then
// the 32 lane sums added in lane order.  Every kernel that sums these columns
// uses this one order, so their floats agree bit for bit.
constexpr int kWarpColumnMaxE = 32;

__device__ __forceinline__ float warp_column_sum(const float* __restrict__ m, int nrows, int ld, int col) {
    const int lane = threadIdx.x & 31;
    float s = 0.f;
#pragma unroll 4
    for (int b = lane; b < nrows; b += 32) s += __ldg(m + (size_t)b * ld + col);
    float tot = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) tot += __shfl_sync(0xffffffffu, s, j);
    return tot;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Arg-max over a warp with ties resolved to the lower index; every lane gets
// the winner.  Lanes with idx < 0 hold no candidate.
__device__ __forceinline__ void warp_argmax(float& v, int& idx) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, o);
        int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        bool take = (oi >= 0) && (idx < 0 || ov > v || (ov == v && oi < idx));
        if (take) {
            v = ov;
            idx = oi;
        }
    }
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// ---------------------------------------------------------------------------
// Launchers (one per kernel family).  All return cudaError_t of the launch.
// ---------------------------------------------------------------------------

// Fused router for E <= kWarpRouterMaxE: logits, softmax, top-k, gates, a
// per-block partial sum of the softmax rows (p_part [nblk][E]) and, when
// block_hist != nullptr, the per-block expert histogram of the chosen ids
// (block_hist [nblk][E]); when probs != nullptr, every softmax row (probs
// [T][E]).  k = 0 computes the softmax only (no ids, no gates).
cudaError_t launch_router_warp(int dtype, int T, int d, int E, int k, const void* x, const void* w_gate,
                               const float* logit_bias, const float* select_bias, int renormalize,
                               int32_t* topk_ids, float* gates, float* p_part, int32_t* block_hist,
                               cudaStream_t s, float* probs = nullptr);

// Router for T <= kSplitDRouterMaxT and E <= 32: one block per token, same
// outputs with one histogram row per token.
// group != nullptr (T <= 256, E <= 32): the last block to finish also groups
// the batch into *group (as launch_group_scan with one token per histogram
// row, statistics included when group->p_part is set); `counter` is a
// workspace word that is zero before the launch and zero again after it.
struct GroupOut;
cudaError_t launch_router_split_d(int dtype, int T, int d, int E, int k, const void* x, const void* w_gate,
                                  const float* logit_bias, const float* select_bias, int renormalize,
                                  int32_t* topk_ids, float* gates, float* p_part, int32_t* block_hist,
                                  cudaStream_t s, float* probs = nullptr, const GroupOut* group = nullptr,
                                  int capacity = -1, unsigned int* counter = nullptr, int* status = nullptr);

// Softmax / top-k over precomputed fp32 logits [T][E] (any E <= kMaxExperts);
// same outputs as the fused router.
// nsplit > 1: logits holds nsplit fp32 K slices [nsplit][T][E] of the
// logits GEMM, added in slice order.
cudaError_t launch_router_from_logits(int T, int E, int k, const float* logits, const float* logit_bias,
                                      const float* select_bias, int renormalize, int32_t* topk_ids,
                                      float* gates, float* p_part, int32_t* block_hist, cudaStream_t s,
                                      float* probs = nullptr, int nsplit = 1);

// p_mean[e] = (sum over blocks of p_part[b][e]) / T, fixed order.
cudaError_t launch_p_mean(int T, int E, int nblk, const float* p_part, float* p_mean, cudaStream_t s);

// Expert histogram of topk_ids per chunk of `chunk` tokens.
cudaError_t launch_group_hist(int T, int E, int k, int chunk, const int32_t* topk_ids, int32_t* block_hist,
                              int* status, cudaStream_t s);

struct GroupOut {
    int32_t* counts;
    int32_t* kept;
    int32_t* offsets;
    int32_t* sorted_token_ids;
    int32_t* slot_pos;
    float* gates_perm;
    int32_t* n_dropped;
    // optional load statistics, written by block 0 when p_part != nullptr
    const float* p_part;
    int p_nblk;
    float* f;
    float* p_mean;
    float* L;
    float alpha;
};

// Scan of the block histograms, stable ranks, capacity cut, permutation.
// block_hist holds one row per chunk of `chunk` tokens.
cudaError_t launch_group_scan(int T, int E, int k, int chunk, int capacity, const int32_t* topk_ids,
                              const float* gates, const int32_t* block_hist, const GroupOut& o, int* status,
                              cudaStream_t s);

// x_perm[pos] = x[sorted_token_ids[pos]] for pos < offsets[E].
cudaError_t launch_gather_rows(int dtype, int T, int d, int rows_max, const int32_t* offsets_end,
                               const int32_t* sorted_token_ids, const void* x, void* x_perm, int* status,
                               cudaStream_t s);

// y[t] = sum_j y_perm[slot_pos[t][j]] (slot_pos >= 0) + y_shared[t]; the
// rows are fp32, or bf16 when rows_bf16.
cudaError_t launch_combine(int dtype, int T, int d, int k, const void* y_perm, const int32_t* slot_pos,
                           const void* y_shared, void* y, cudaStream_t s, int32_t* n_empty = nullptr,
                           bool rows_bf16 = false);

// Expert-choice routing: expert e takes the C tokens with the largest
// probs[t][e] (ties to the lower token index), in ascending token order, as
// rows [e*C, (e+1)*C) of the permuted layout; writes sorted_token_ids and
// gates_perm [E*C], slot_pos [T][E] (row or -1), counts/kept [E] (= C,
// nullable), offsets [E+1] (= e*C) and zeroes *n_empty (nullable).
cudaError_t launch_ec_select(int T, int E, int C, const float* probs, int32_t* sorted_token_ids, float* gates_perm,
                             int32_t* slot_pos, int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* n_empty,
                             cudaStream_t s);

// bias[e] -= gamma * sign(counts[e] - T k / E).
cudaError_t launch_bias_update(int T, int E, int k, const int32_t* counts, float gamma, float* bias, cudaStream_t s);

// f = counts/(T k), L = alpha E sum f p.
cudaError_t launch_load_stats(int T, int E, int k, float alpha, const int32_t* counts, const float* p_mean,
                              float* f, float* L, cudaStream_t s);

// ---- grouped GEMMs ----------------------------------------------------------

enum GemmMode : int {
    kGemmSwiGLU = 0,  // out(dtype) = silu(A W1^T) * (A W3^T), N = F columns
    kGemmScale = 1,   // out(fp32)  = row_scale[row] * (A B^T)  (row_scale may be null: 1)
    kGemmPlain = 2,   // out(fp32)  = A B^T
    kGemmScaleSplit = 3,  // out(fp32) = row_scale[row] * ((A + A2) B^T), A and A2 bf16 (hi and lo halves)
    kGemmSwigluBwd = 4,   // D = A B^T consumed in the epilogue by the SwiGLU backward (bwd_* fields)
};

// One grouped problem: rows of A are split into groups by offsets (G+1
// entries, device) or form a single group of M rows when offsets is null.
// Group g multiplies its rows by B rows [g*N, (g+1)*N) (B is [G*N][K]).
struct GemmProblem {
    const void* A;        // [rows][K]
    int a_rows;           // allocated rows of A (bounds the loads)
    const void* B1;       // [G*N][K]
    const void* B2;       // SwiGLU only: W3 with B1's layout
    const int32_t* offsets;
    int G;
    int M;                // rows when offsets == nullptr
    int N;
    int K;
    void* out;            // [rows][N]
    int out_bf16;         // Scale / ScaleSplit modes: out holds bf16 rows (else fp32)
    const float* row_scale;
    const void* A2;       // kGemmScaleSplit: the lo half of A, same layout
    void* out2;           // kGemmSwiGLU: optional lo half of H (H - bf16(H)), same layout as out
    float* part;          // split-K: fp32 partials [ksplit][a_rows][2N (SwiGLU) or N]
    const int32_t* a_gather;  // non-null: A row r is row a_gather[r] of A, which has a_src_rows rows
    int a_src_rows;
    // FP8 (E4M3) weights (launch_gemm_tc_w8): B1/B2 hold one-byte codes and
    // these the fp32 scale of every weight row ([G*N]), applied per column
    const float* wscale1;
    const float* wscale2;
    // FP8 tokens (launch_gemm_decode with w8): A holds the hi and A2 the lo
    // E4M3 codes of every token row, a_scale its power-of-two scale (indexed
    // like the rows of A, or of the gather source), A row = a_scale * (hi + lo)
    const float* a_scale;
    // K-grouped problem (launch_gemm_tc, ksplit 1, no offsets; Plain mode, or
    // Scale mode without row scales on CTA pairs): group g
    // multiplies A rows [0, M) by B rows [0, N) over the K window
    // [kbase[g], kbase[g] + klen[g]) and writes output rows g*M .. g*M + M - 1
    // (weight gradients: a contraction over each expert's token rows)
    const int32_t* kbase;
    const int32_t* klen;
    // MN-major B (launch_gemm_tc, Plain / Scale modes, ksplit 1, plain A): B1
    // holds B^T per group, [G][K][N] (N a multiple of 8), read without a
    // transposed copy.  kpart > 0: K = 2 kpart in two parts, A = [rows][2 kpart]
    // (part 0 then part 1 of every row), B1 = part 0 of B^T [G][kpart][N], B2
    // = part 1; each part is padded to whole 64-deep k-blocks with zeros.
    int b_mn;
    int kpart;
    // kGemmSwiGLU (launch_gemm_tc, bf16 weights, ksplit 1): when non-null, the
    // fp32 pre-activations G = A W1^T and U = A W3^T [rows][N] are written too
    float* out_g;
    float* out_u;
    // kGemmSwigluBwd (launch_gemm_tc, ksplit 1): the product D = A B^T [rows][N]
    // is not stored; with G, U the recomputed up projections [rows][N] fp32 and
    // g = row_scale[row] (null: 1), the epilogue writes per element
    //   h = silu(G) U,  dh = g D,  dG = dh U silu'(G),  dU = dh silu(G)
    // as bf16 dGU [rows][2N] (dG, then dU) and Hb = bf16(h) [rows][N], and, per
    // 256-column tile n, dgp_part[n * dgp_ld + row] = sum over its columns of D h
    const float* bwd_G;
    const float* bwd_U;
    void* bwd_dGU;
    void* bwd_Hb;
    float* bwd_dgp_part;
    int bwd_dgp_ld;
};

// Tensor-core (tcgen05) path, bf16 operands, fp32 accumulate.  Runs up to two
// problems (a routed one and a shared-expert one) in one persistent launch.
// ksplit > 1 splits every tile's K range into ksplit slices that write fp32
// partials to GemmProblem::part instead of `out` (finish with
// launch_swiglu_finalize or the split-aware combine / reduce).
// pair = true runs the 2-SM kernel (256-row tiles on CTA pairs; SwiGLU and
// Scale modes, ksplit 1, plain A) for large expert segments.
cudaError_t launch_gemm_tc(int mode, const GemmProblem* probs, int nprob, int* status, int num_sms,
                           cudaStream_t s, int ksplit = 1, bool pair = false);

// Failure-detection test switch (moe_test_stall_gemm): when set, the
// tensor-core GEMM launchers make the producer issue no loads and bound every
// wait at kStallWaitLimitNs, so the kernels report MOE_ERR_TIMEOUT and return.
bool test_stall_gemm();
constexpr uint64_t kStallWaitLimitNs = 20000000ull;  // 20 ms

// Same grouped GEMM with FP8 (E4M3) B operands: raw one-byte tiles stream in
// through a deep TMA ring, four converter warps widen them (exactly) to the
// bf16 swizzled layout the MMA reads, and the epilogue multiplies column n by
// wscale[n] (per weight row).  SwiGLU and Scale modes, 1-CTA tiles, split-K
// and gathered A as in launch_gemm_tc; K must be a multiple of 16.
cudaError_t launch_gemm_tc_w8(int mode, const GemmProblem* probs, int nprob, int* status, int num_sms,
                              cudaStream_t s, int ksplit = 1);

// Decode-sized batches: the same grouped GEMM with the weights on the MMA's M
// side (D^T = W X^T; nt = 32 or 64 token rows per tile, or 48 with FP8
// weights, which keeps five stages in flight), bf16 or FP8 (w8)
// weights, SwiGLU and Scale modes, split-K and gathered token rows; no split H.
// balanced (ksplit 2, one problem): every CTA takes an equal contiguous
// share of all tiles' k-blocks (slice 0 = a tile's part from k-block 0,
// slice 1 = the rest, zeros when one CTA covered the whole tile).
// tile_sync (SwiGLU, ksplit > 1): one zeroed counter per output tile
// (decode_tile_sync_words); the kernel then finishes the SwiGLU itself (no
// launch_swiglu_finalize) and leaves the counters zero again.
cudaError_t launch_gemm_decode(int mode, const GemmProblem* probs, int nprob, int* status, int num_sms,
                               cudaStream_t s, int ksplit, bool w8, int nt, bool balanced = false,
                               unsigned int* tile_sync = nullptr);

// ---- backward pass (backward.cu) ----
// kbase[e] = sum_{e' < e} round64(klen[e']), klen[e] = offsets[e+1] - offsets[e];
// const_len >= 0: one window of const_len rows, writing offsets = {0, const_len}.
cudaError_t launch_k_windows(int E, int32_t* offsets, int32_t* kbase, int32_t* klen, int const_len, cudaStream_t s);
// bf16 rows of expert e (src rows offsets[e] + k, columns col0 .. col0 + C - 1,
// times row_scale[row] when given) -> dst[c][kbase[e] + k], zero-filled to
// the next multiple of 64; ncols = columns of dst to cover.
cudaError_t launch_transpose_windows(const void* src, size_t ld_src, int col0, int C, int E, const int32_t* offsets,
                                     const int32_t* kbase, const int32_t* klen, const float* row_scale, void* dst,
                                     size_t ld_dst, int ncols, cudaStream_t s);
// dlogits [T][E] from the gate gradients (via slot_pos) and the balance loss.
cudaError_t launch_router_backward(int T, int E, int k, const float* probs, const int32_t* ids,
                                   const int32_t* slot_pos, const float* gates, const float* dgp, int renormalize,
                                   const int32_t* counts, float alpha, float dL, float* dlogits, cudaStream_t s);
// R[t] = dlogits[t] W_g (+ extra[t]).
cudaError_t launch_router_dx(int dtype, int T, int E, int d, const float* dlogits, const void* w_gate,
                             const float* extra, float* R, cudaStream_t s);
// part[s][e][i] = sum over token chunk s of dlogits[t][e] x[t][i].
// Token chunks launch_wgate_grad is given for E experts and d columns (the
// partial buffer holds that many [E][d] slices).
int wgate_grad_split(int E, int d);
cudaError_t launch_wgate_grad(int dtype, int T, int E, int d, const float* dlogits, const void* x, int nsplit,
                              float* part, cudaStream_t s);

// Per-row E4M3 quantisation of a [rows][cols] bf16 or fp32 matrix (cols a
// multiple of 16): q [rows][cols] codes, scale [rows] fp32.
cudaError_t launch_quantize_fp8(int dtype, long long rows, int cols, const void* w, uint8_t* q, float* scale,
                                cudaStream_t s);

// bf16 rows (K a multiple of 8) -> E4M3 hi and lo code rows [rows][K] and a
// power-of-two scale per row, row = scale * (hi + lo) (exact for entries
// within 2^10 of the row's largest magnitude).  Output row r is row
// gather[r] of x ([x_rows][K]) when gather is given, else row r; rows at or
// beyond *live_rows (nullable) are skipped.  Feeds the FP8 tensor-core path
// of the decode GEMM.
cudaError_t launch_split_e4m3(int rows, int K, const void* x, int x_rows, const int32_t* gather,
                              const int32_t* live_rows, uint8_t* hi, uint8_t* lo, float* scale, cudaStream_t s);

// H[r][f] = silu(sum_s P[s][r][f]) * sum_s P[s][r][N + f] (bf16, and the lo
// half when h_lo != nullptr) for r < rows, rows = *rows_dev when non-null.
cudaError_t launch_swiglu_finalize(int rows_max, const int32_t* rows_dev, int N, int ksplit, const float* part,
                                   void* h, void* h_lo, cudaStream_t s);

// out[r][c] = sum_s P[s][r][c] for r < rows (rows_dev as above), stored as
// fp32 or, with out_bf16, rounded to bf16.
cudaError_t launch_reduce_partials(int rows_max, const int32_t* rows_dev, int N, int ksplit, const float* part,
                                   void* out, cudaStream_t s, bool out_bf16 = false);

// Combine over split-K partials: y[t] = sum_j (sum_s Yp[s][pos_j]) + sum_s Ys[s][t];
// round_rows rounds each entry's slice sum to bf16 before adding it (the
// layer keeps its rows in bf16).
cudaError_t launch_combine_split(int dtype, int T, int d, int k, const float* y_perm, size_t perm_stride,
                                 int nsplit, const int32_t* slot_pos, const float* y_shared, size_t shared_stride,
                                 int shared_nsplit, void* y, cudaStream_t s, int32_t* n_empty = nullptr,
                                 bool round_rows = false);

// CUDA-core fp32 path with the same semantics (dtype MOE_F32).
cudaError_t launch_gemm_simt_f32(int mode, const GemmProblem* probs, int nprob, cudaStream_t s);

// ---- decode_fused.cu: the whole token-choice layer for batches of at most
// kFusedMaxT tokens on routers of at most kFusedMaxE experts, in two launches
// (router + up projection + SwiGLU; down projection + gates + shared expert).
constexpr int kFusedMaxT = 1;
constexpr int kFusedMaxE = 32;
constexpr int kFusedMaxEntries = 16;  // T k routing decisions

struct FusedDecodeArgs {
    int T, d, E, k, F, Fs, n_shared, renormalize, capacity, y_fp32, fp8;
    float alpha;
    const void *x, *wg;                           // bf16 [T][d], [E][d]
    const float *logit_bias, *select_bias;        // [E], nullable
    const void *w1, *w3, *w2, *ws1, *ws3, *ws2;   // bf16 weights or E4M3 codes
    const float *s1, *s3, *s2, *ss1, *ss3, *ss2;  // FP8 row scales (fp8 = 1)
    void *h, *h_shared;                           // bf16 H [T k][F], [T][Fs] (workspace)
    void* y;                                      // [T][d] bf16, or fp32 when y_fp32
    int32_t *counts, *kept, *n_dropped;           // statistics, each nullable
    float *f, *p, *L;
    int* status;
};

// Shared-memory and grid plan of the two kernels for one layer; ok is false
// when the layer is not one they take (routing, dtype, sizes) or does not fit.
struct FusedPlan {
    bool ok;
    int up_rows, up_wslice, up_stages;      // a stage: up_rows whole W1 and W3 rows; d elements per consumer warp
    int dn_wslice, dn_wslice_s, dn_stages;  // per consumer warp: F (F_s) elements of each W2 row
    int dn_rows_stage;                      // a stage: this many whole consecutive W2 rows (1 or 2)
    int up_pv, dn_pv;                       // activation vectors per lane and token (2 or 4)
    int dn_rows, dn_cols;                   // output channels per CTA (at most); partial columns (at most)
    int grid_up, grid_dn;
    size_t up_part_bytes, up_smem;                   // partial dots, then the ring
    size_t dn_stage_bytes, dn_part_bytes, dn_smem;   // partial dots, then the ring
};
FusedPlan fused_decode_plan(const moe_config& c, bool fp8, int sms);
cudaError_t launch_fused_up(const FusedDecodeArgs& a, const FusedPlan& p, cudaStream_t s);
cudaError_t launch_fused_down(const FusedDecodeArgs& a, const FusedPlan& p, cudaStream_t s);

}  // namespace moe
