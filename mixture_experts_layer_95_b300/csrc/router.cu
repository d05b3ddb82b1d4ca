// router.cu -- router logits, softmax, top-k and gates.
//
// Computes, per token t (sources: "Mixture of Experts" notes, How it works:
// g(x) = softmax(W_g x), keep the top-k, renormalise; "MoE Architecture" s2
// Gating Function; "Mixture of experts (MoE)" handbook, Load balancing: the
// per-expert bias is added to the routing score for the choice only):
//   l_e = <W_g[e], x_t> + logit_bias[e]           (fp32 accumulate)
//   p   = softmax(l)
//   ids = top-k of l + select_bias, descending, ties to the lower index
//   g_j = p[ids_j] / sum_j p[ids_j]   (or p[ids_j] without renormalisation)
// plus, per block, the partial column sums of p (for the mean router
// probability p_i) and the histogram of the chosen ids (for the grouping scan),
// and optionally the whole row p (expert-choice routing ranks tokens by it;
// it then calls the router with k = 0, which skips the top-k).
//
// Three kernels:
//  * router_warp_kernel -- one warp per token, E <= 16 experts, W_g staged in
//    shared memory.  Each lane streams 16-byte vectors of x, keeps E fp32
//    partial dots in registers and finishes them with butterfly shuffles;
//    afterwards lane e owns expert e.
//  * router_split_d_kernel -- decode-sized batches: one block per token.
//  * router_logits_kernel -- softmax/top-k over fp32 logits produced by a
//    tensor-core GEMM (large E); lane owns experts lane, lane+32, ...
#include <float.h>

#include <type_traits>

#include "common.cuh"
#include "route_math.cuh"

namespace moe {
namespace {
using namespace route_math;

// softmax / top-k pass over precomputed logits: 16 warps share a block's 64
// tokens (8 when each lane holds 32 experts' logits), so that a top-8 over 256
// experts (k sequential warp reductions per token) keeps enough warps in flight
template <int NJ>
constexpr int logits_warps() {
    return NJ >= 32 ? 8 : 16;
}

// Writes the per-block partial sums of p and the per-block id histogram.
template <int NJ, int NW>
__device__ __forceinline__ void block_epilogue(int E, const float (&psum)[NJ], const int (&hcnt)[NJ],
                                               float* p_part, int32_t* block_hist, float* s_p, int* s_h) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int e = lane + 32 * j;
        if (e < E) {
            s_p[warp * E + e] = psum[j];
            s_h[warp * E + e] = hcnt[j];
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float ps = 0.f;
        int hs = 0;
        for (int w = 0; w < NW; ++w) {  // fixed order: deterministic
            ps += s_p[w * E + e];
            hs += s_h[w * E + e];
        }
        if (p_part) p_part[(size_t)blockIdx.x * E + e] = ps;
        if (block_hist) block_hist[(size_t)blockIdx.x * E + e] = hs;
    }
}

// Fused router for E <= NE.  W_g is copied once per block into shared memory
// (rows E..NE-1 zero-filled, so the inner loop has no branches).  Each warp
// owns kTpw consecutive tokens and works on all of them at once: every
// 16-byte vector of W_g read from shared memory feeds kTpw tokens, and the x
// vectors of all kTpw tokens are in flight together.  Lanes accumulate NE fp32
// partial dots per token, finished with butterfly shuffles.
template <typename T, int NE>
__global__ void __launch_bounds__(kWarpRouterThreads) router_warp_kernel(
    int Tn, int d, int E, int k, const T* __restrict__ x, const T* __restrict__ wg,
    const float* __restrict__ logit_bias, const float* __restrict__ select_bias, int renormalize,
    int32_t* __restrict__ topk_ids, float* __restrict__ gates, float* __restrict__ p_part,
    int32_t* __restrict__ block_hist, float* __restrict__ probs) {
    pdl_wait();
    constexpr int kW = kWarpRouterThreads / 32;
    constexpr int kTpw = kWarpRouterChunk / kW;
    constexpr int VE = Vec<T>::kElems;
    extern __shared__ uint4 s_w[];  // [NE][d / VE] 16-byte vectors
    __shared__ float s_p[kW * NE];
    __shared__ int s_h[kW * NE];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = d / VE;  // vectors per row
    {
        const uint4* src = reinterpret_cast<const uint4*>(wg);
#pragma unroll 8
        for (int i = threadIdx.x; i < NE * nv; i += blockDim.x)
            s_w[i] = (i < E * nv) ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    const int t0 = blockIdx.x * kWarpRouterChunk + warp * kTpw;
    const uint4* xr[kTpw];
#pragma unroll
    for (int q = 0; q < kTpw; ++q) {
        const int t = t0 + q < Tn ? t0 + q : Tn - 1;  // clamp: rows past T are read but never used
        xr[q] = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    }
    float acc[kTpw][NE];
#pragma unroll
    for (int q = 0; q < kTpw; ++q)
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[q][e] = 0.f;
    // U of the lane's vectors per token are loaded before any is used, so
    // U * kTpw loads are in flight per lane; they are added in the same order
    // (v = lane, lane + 32, ...) as one at a time.  (U = 2 for 16 experts keeps
    // the accumulators within the 128 registers of a 512-thread block.)
    constexpr int U = NE <= 8 ? 4 : 2;
    for (int v0 = lane; v0 < nv; v0 += 32 * U) {
        uint4 raw[U][kTpw];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int q = 0; q < kTpw; ++q)
                raw[u][q] = v0 + 32 * u < nv ? __ldg(xr[q] + v0 + 32 * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 32 * u;
            if (v >= nv) break;  // v rises with u
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                // bf16 pairs straight into mixed-precision FMAs: the same sums
                // as widening both operands, element by element in order
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    const uint4 w4 = s_w[e * nv + v];
                    const uint32_t wd[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int q = 0; q < kTpw; ++q) {
                        const uint32_t xd[4] = {raw[u][q].x, raw[u][q].y, raw[u][q].z, raw[u][q].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[q][e] = fma2_bf16(xd[j], wd[j], acc[q][e]);
                    }
                }
            } else {
                float xv[kTpw][VE];
#pragma unroll
                for (int q = 0; q < kTpw; ++q) widen(raw[u][q], xv[q], static_cast<const T*>(nullptr));
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    float wv[VE];
                    widen(s_w[e * nv + v], wv, static_cast<const T*>(nullptr));
#pragma unroll
                    for (int q = 0; q < kTpw; ++q)
#pragma unroll
                        for (int i = 0; i < VE; ++i) acc[q][e] = fmaf(xv[q][i], wv[i], acc[q][e]);
                }
            }
        }
    }
    float psum[1] = {0.f};
    int hcnt[1] = {0};
#pragma unroll
    for (int q = 0; q < kTpw; ++q) {
        if (t0 + q >= Tn) break;  // warp-uniform
        float l[1] = {-FLT_MAX};
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            const float v = warp_sum(acc[q][e]);
            if (lane == e && e < E) l[0] = v + (logit_bias ? __ldg(logit_bias + e) : 0.f);
        }
        softmax_topk<1>(t0 + q, E, k, l, select_bias, renormalize, topk_ids, gates, psum, hcnt, probs);
    }
    block_epilogue<1, kW>(E, psum, hcnt, p_part, block_hist, s_p, s_h);
    __syncthreads();
    pdl_trigger();  // after this block's last global write
}

// Grouping of a decode-sized batch inside the router launch (T <= 256,
// E <= 32): the last router block to finish -- every block counts itself in
// on a workspace counter after its writes, so the one that sees the count
// reach the grid size knows every token is routed -- groups all T k entries
// ("Mixture of experts (MoE)" handbook, Implementation: stable sort by
// expert, counts, running starts; capacity as in the notes and "MoE
// Architecture" s2) and writes the load statistics, which saves the separate
// grouping launch and its dependency wait.  A token picks each expert at most
// once, so an entry's rank inside its expert is the number of earlier tokens
// that picked that expert: a prefix sum down one column of the per-token id
// histogram.  Results equal group_scan_kernel's bit for bit (integers; the
// statistics add in the same order).
struct SmallGroup {
    GroupOut o;
    int capacity;
    unsigned int* counter;  // zero before the launch; wraps back to zero after it
    int* status;
};

constexpr int kSmallGroupMaxT = kSplitDRouterMaxT;
constexpr int kSmallGroupMaxE = 32;

// Same order of additions as warp_column_sum, through L2 (the rows were
// written by other blocks of this launch).
__device__ __forceinline__ float warp_column_sum_cg(const float* m, int nrows, int ld, int col) {
    const int lane = threadIdx.x & 31;
    float s = 0.f;
#pragma unroll 4
    for (int b = lane; b < nrows; b += 32) s += __ldcg(m + (size_t)b * ld + col);
    float tot = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) tot += __shfl_sync(0xffffffffu, s, j);
    return tot;
}

// Runs in one block of kSplitDThreads threads.  ids, gates [T][k], hist and
// p_part [T][E] hold every token's row.
__device__ void group_small_batch(const SmallGroup& g, int Tn, int E, int k, const int32_t* ids, const float* gates,
                                  const int32_t* hist, const float* p_part) {
    __shared__ int s_rank[kSmallGroupMaxT][kSmallGroupMaxE];  // earlier tokens that picked each expert
    __shared__ int s_cnt[kSmallGroupMaxE], s_off[kSmallGroupMaxE + 1];
    __shared__ float s_fp[kSmallGroupMaxE];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kW = kSplitDThreads / 32;
    const int n = Tn * k;
    // 1. per expert: exclusive prefix of its histogram column over tokens
    //    (lane l owns tokens [8 l, 8 l + 8))
    for (int e = warp; e < E; e += kW) {
        int v[8], loc = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = lane * 8 + i;
            v[i] = t < Tn ? __ldcg(hist + (size_t)t * E + e) : 0;
            loc += v[i];
        }
        int incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int run = incl - loc;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = lane * 8 + i;
            if (t < Tn) s_rank[t][e] = run;
            run += v[i];
        }
        if (lane == 31) s_cnt[e] = incl;
    }
    __syncthreads();
    // 2. capacity cut and expert offsets (warp 0, one lane per expert)
    if (warp == 0) {
        const int cnt = lane < E ? s_cnt[lane] : 0;
        const int kept = (g.capacity >= 0 && cnt > g.capacity) ? g.capacity : cnt;
        int incl = kept;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane < E) {
            s_off[lane] = incl - kept;
            g.o.counts[lane] = cnt;
            g.o.kept[lane] = kept;
            g.o.offsets[lane] = incl - kept;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (lane == 0) {
            s_off[E] = total;
            g.o.offsets[E] = total;
            *g.o.n_dropped = n - total;
        }
    }
    // 3. load statistics: f = counts / (T k), p = mean softmax row, L = alpha E sum f p
    //    (the additions of group_scan_kernel and moe_load_stats, in their order)
    if (g.o.p_part) {
        for (int e = warp; e < E; e += kW) {
            const float ps = warp_column_sum_cg(p_part, Tn, E, e);
            if (lane == 0) {
                const float pm = ps / (float)Tn;
                const float f = (float)s_cnt[e] / ((float)Tn * (float)k);
                if (g.o.p_mean) g.o.p_mean[e] = pm;
                if (g.o.f) g.o.f[e] = f;
                s_fp[e] = f * pm;
            }
        }
    }
    __syncthreads();
    if (g.o.p_part && g.o.L && threadIdx.x == 0) {
        float acc = 0.f;
        for (int e = 0; e < E; ++e) acc += s_fp[e];
        *g.o.L = g.o.alpha * (float)E * acc;
    }
    // 4. positions: entries in flat order; positions past the kept total get
    //    sorted_token_ids = -1, gates_perm = 0
    const int total = s_off[E];
    for (int pos = total + threadIdx.x; pos < n; pos += blockDim.x) {
        g.o.sorted_token_ids[pos] = -1;
        g.o.gates_perm[pos] = 0.f;
    }
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int t = i / k;
        const int e = __ldcg(ids + i);
        int pos = -1;
        if (e < 0 || e >= E) {
            record_status(g.status, kStatusBounds);
        } else {
            const int rank = s_rank[t][e];
            if (g.capacity < 0 || rank < g.capacity) pos = s_off[e] + rank;
            if (pos >= s_off[e + 1]) {  // ids that disagree with the histogram rows
                record_status(g.status, kStatusBounds);
                pos = -1;
            }
        }
        g.o.slot_pos[i] = pos;
        if (pos >= 0) {
            g.o.sorted_token_ids[pos] = t;
            g.o.gates_perm[pos] = __ldcg(gates + i);
        }
    }
}

// Router for decode-sized batches: one block per token, the d dimension split
// over the block's threads (each thread owns 16-byte vectors v = tid,
// tid + 256, ...), W_g read straight from L2/L1.  The E partial dots are
// reduced across the block in a fixed order; warp 0 then runs the shared
// softmax/top-k epilogue.  Histogram and p rows are per token (chunk = 1).
template <typename T, int NE>
__global__ void __launch_bounds__(kSplitDThreads) router_split_d_kernel(
    int Tn, int d, int E, int k, const T* __restrict__ x, const T* __restrict__ wg,
    const float* __restrict__ logit_bias, const float* __restrict__ select_bias, int renormalize,
    int32_t* __restrict__ topk_ids, float* __restrict__ gates, float* __restrict__ p_part,
    int32_t* __restrict__ block_hist, float* __restrict__ probs, const SmallGroup group) {
    pdl_wait();
    constexpr int VE = Vec<T>::kElems;
    constexpr int kW = kSplitDThreads / 32;
    __shared__ float s_red[kW][NE];
    __shared__ int s_last;
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = d / VE;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const uint4* w = reinterpret_cast<const uint4*>(wg);
    float acc[NE];
#pragma unroll
    for (int e = 0; e < NE; ++e) acc[e] = 0.f;
    for (int v = threadIdx.x; v < nv; v += kSplitDThreads) {
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {  // (the same sums as widening, in order)
            const uint4 x4 = __ldg(xr + v);
            const uint32_t xd[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
            for (int e = 0; e < NE; ++e) {
                if (e < E) {
                    const uint4 w4 = __ldg(w + (size_t)e * nv + v);
                    const uint32_t wd[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[e] = fma2_bf16(xd[j], wd[j], acc[e]);
                }
            }
        } else {
            float xv[VE];
            widen(__ldg(xr + v), xv, static_cast<const T*>(nullptr));
#pragma unroll
            for (int e = 0; e < NE; ++e) {
                if (e < E) {
                    float wv[VE];
                    widen(__ldg(w + (size_t)e * nv + v), wv, static_cast<const T*>(nullptr));
#pragma unroll
                    for (int i = 0; i < VE; ++i) acc[e] = fmaf(xv[i], wv[i], acc[e]);
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        const float v = warp_sum(acc[e]);
        if (lane == 0) s_red[warp][e] = v;
    }
    __syncthreads();
    if (warp == 0) {
        float l[1] = {-FLT_MAX};
        if (lane < E) {
            float v = 0.f;
            for (int q = 0; q < kW; ++q) v += s_red[q][lane];  // fixed order
            l[0] = v + (logit_bias ? __ldg(logit_bias + lane) : 0.f);
        }
        float psum[1] = {0.f};
        int hcnt[1] = {0};
        softmax_topk<1>(t, E, k, l, select_bias, renormalize, topk_ids, gates, psum, hcnt, probs);
        if (lane < E) {
            if (p_part) p_part[(size_t)t * E + lane] = psum[0];
            if (block_hist) block_hist[(size_t)t * E + lane] = hcnt[0];
        }
    }
    if (group.counter == nullptr) return;  // routing only
    // count this block in after its writes; the last one groups the batch
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicInc(group.counter, gridDim.x - 1) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    group_small_batch(group, Tn, E, k, topk_ids, gates, block_hist, p_part);
}

template <int NJ>
__global__ void __launch_bounds__(32 * logits_warps<NJ>()) router_logits_kernel(
    int Tn, int E, int k, const float* __restrict__ logits, const float* __restrict__ logit_bias,
    const float* __restrict__ select_bias, int renormalize, int32_t* __restrict__ topk_ids,
    float* __restrict__ gates, float* __restrict__ p_part, int32_t* __restrict__ block_hist,
    float* __restrict__ probs, int nsplit) {
    pdl_wait();
    extern __shared__ float s_dyn[];
    float* s_p = s_dyn;
    constexpr int kW = logits_warps<NJ>();
    constexpr int kTokensPerWarp = kRouterTokensPerBlock / kW;
    int* s_h = reinterpret_cast<int*>(s_dyn + kW * E);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float psum[NJ];
    int hcnt[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        psum[j] = 0.f;
        hcnt[j] = 0;
    }
    // the logits of kPre tokens at a time (at most 64 registers) are loaded
    // before their softmax / top-k, so the warp waits for memory once per
    // group instead of once per token
    constexpr int kPre = kTokensPerWarp * NJ <= 64 ? kTokensPerWarp : (64 / NJ > 0 ? 64 / NJ : 1);
    for (int i0 = 0; i0 < kTokensPerWarp; i0 += kPre) {
        const int t0 = blockIdx.x * kRouterTokensPerBlock + warp * kTokensPerWarp + i0;
        if (t0 >= Tn) break;
        float l[kPre][NJ];
#pragma unroll
        for (int i = 0; i < kPre; ++i)
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int e = lane + 32 * j;
                l[i][j] = (t0 + i < Tn && e < E) ? logits[(size_t)(t0 + i) * E + e] : -FLT_MAX;
            }
        for (int sl = 1; sl < nsplit; ++sl)  // the logits GEMM's K slices, added in slice order
#pragma unroll
            for (int i = 0; i < kPre; ++i)
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int e = lane + 32 * j;
                    if (t0 + i < Tn && e < E) l[i][j] += logits[((size_t)sl * Tn + t0 + i) * E + e];
                }
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
            if (i0 + i >= kTokensPerWarp || t0 + i >= Tn) break;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int e = lane + 32 * j;
                if (e < E) l[i][j] += logit_bias ? __ldg(logit_bias + e) : 0.f;
            }
            softmax_topk<NJ>(t0 + i, E, k, l[i], select_bias, renormalize, topk_ids, gates, psum, hcnt, probs);
        }
    }
    block_epilogue<NJ, kW>(E, psum, hcnt, p_part, block_hist, s_p, s_h);
    __syncthreads();
    pdl_trigger();
}

// Column means of the router's p rows, in the order the fused grouping scan
// sums them (warp_column_sum for small E, row order otherwise).
__global__ void p_mean_kernel(int Tn, int E, int nblk, const float* __restrict__ p_part, float* __restrict__ p_mean) {
    pdl_wait();
    if (E <= kWarpColumnMaxE) {
        const int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // one warp per expert
        if (e >= E) return;
        const float s = warp_column_sum(p_part, nblk, E, e);
        if ((threadIdx.x & 31) == 0) p_mean[e] = Tn > 0 ? s / (float)Tn : 0.f;
        return;
    }
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    float s = 0.f;
    for (int b = 0; b < nblk; ++b) s += p_part[(size_t)b * E + e];
    p_mean[e] = Tn > 0 ? s / (float)Tn : 0.f;
}

}  // namespace

cudaError_t launch_router_warp(int dtype, int T, int d, int E, int k, const void* x, const void* w_gate,
                               const float* logit_bias, const float* select_bias, int renormalize,
                               int32_t* topk_ids, float* gates, float* p_part, int32_t* block_hist,
                               cudaStream_t s, float* probs) {
    const int nblk = (T + kWarpRouterChunk - 1) / kWarpRouterChunk;
    if (nblk == 0) return cudaSuccess;
    const int ne = warp_router_width(E);
    const size_t smem = warp_router_smem_bytes(E, d, dtype);
    const dim3 grid(nblk), block(kWarpRouterThreads);
#define MOE_ROUTER_CASE(TY, NE)                                                                                 \
    do {                                                                                                        \
        cudaError_t e_ = cudaFuncSetAttribute(router_warp_kernel<TY, NE>,                                       \
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);          \
        if (e_ != cudaSuccess) return e_;                                                                       \
        launch_pdl(router_warp_kernel<TY, NE>, dim3(grid), dim3(block), smem, s, T, d, E, k, static_cast<const TY*>(x),           \
                                                             static_cast<const TY*>(w_gate), logit_bias,       \
                                                             select_bias, renormalize, topk_ids, gates, p_part, \
                                                             block_hist, probs);                                \
    } while (0)
    if (dtype == MOE_BF16) {
        if (ne == 8) MOE_ROUTER_CASE(__nv_bfloat16, 8);
        else MOE_ROUTER_CASE(__nv_bfloat16, 16);
    } else {
        if (ne == 8) MOE_ROUTER_CASE(float, 8);
        else MOE_ROUTER_CASE(float, 16);
    }
#undef MOE_ROUTER_CASE
    return cudaGetLastError();
}

cudaError_t launch_router_split_d(int dtype, int T, int d, int E, int k, const void* x, const void* w_gate,
                                  const float* logit_bias, const float* select_bias, int renormalize,
                                  int32_t* topk_ids, float* gates, float* p_part, int32_t* block_hist,
                                  cudaStream_t s, float* probs, const GroupOut* group, int capacity,
                                  unsigned int* counter, int* status) {
    if (T == 0) return cudaSuccess;
    SmallGroup sg{};
    if (group) {
        // grouping in the last block: every token's ids, gates, p row and histogram row are needed
        if (!counter || !block_hist || !p_part || !topk_ids || !gates || T > kSmallGroupMaxT || E > kSmallGroupMaxE)
            return cudaErrorInvalidValue;
        sg.o = *group;
        sg.capacity = capacity;
        sg.counter = counter;
        sg.status = status;
    }
#define MOE_SPLITD_CASE(TY, NE)                                                                              \
    launch_pdl(router_split_d_kernel<TY, NE>, dim3(T), dim3(kSplitDThreads), 0, s, T, d, E, k, static_cast<const TY*>(x),       \
                                                               static_cast<const TY*>(w_gate), logit_bias,  \
                                                               select_bias, renormalize, topk_ids, gates,  \
                                                               p_part, block_hist, probs, sg)
    if (dtype == MOE_BF16) {
        if (E <= 8) MOE_SPLITD_CASE(__nv_bfloat16, 8);
        else if (E <= 16) MOE_SPLITD_CASE(__nv_bfloat16, 16);
        else MOE_SPLITD_CASE(__nv_bfloat16, 32);
    } else {
        if (E <= 8) MOE_SPLITD_CASE(float, 8);
        else if (E <= 16) MOE_SPLITD_CASE(float, 16);
        else MOE_SPLITD_CASE(float, 32);
    }
#undef MOE_SPLITD_CASE
    return cudaGetLastError();
}

cudaError_t launch_router_from_logits(int T, int E, int k, const float* logits, const float* logit_bias,
                                      const float* select_bias, int renormalize, int32_t* topk_ids,
                                      float* gates, float* p_part, int32_t* block_hist, cudaStream_t s,
                                      float* probs, int nsplit) {
    if (nsplit < 1) return cudaErrorInvalidValue;
    const int nblk = (T + kRouterTokensPerBlock - 1) / kRouterTokensPerBlock;
    if (nblk == 0) return cudaSuccess;
    const dim3 grid(nblk);
#define MOE_LOGITS_CASE(NJ)                                                                                  \
    do {                                                                                                     \
        const size_t smem = (size_t)logits_warps<NJ>() * E * (sizeof(float) + sizeof(int));                 \
        const dim3 block(32 * logits_warps<NJ>());                                                           \
        if (smem > 48 * 1024)                                                                                \
            cudaFuncSetAttribute(router_logits_kernel<NJ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        launch_pdl(router_logits_kernel<NJ>, dim3(grid), dim3(block), smem, s, T, E, k, logits, logit_bias, select_bias,       \
                                                           renormalize, topk_ids, gates, p_part, block_hist, probs, \
                                                           nsplit);                                          \
    } while (0)
    if (E <= 64) MOE_LOGITS_CASE(2);
    else if (E <= 256) MOE_LOGITS_CASE(8);
    else MOE_LOGITS_CASE(32);
#undef MOE_LOGITS_CASE
    return cudaGetLastError();
}

cudaError_t launch_p_mean(int T, int E, int nblk, const float* p_part, float* p_mean, cudaStream_t s) {
    const int threads = E <= kWarpColumnMaxE ? 32 * E : E;
    launch_pdl(p_mean_kernel, dim3((threads + 255) / 256), dim3(256), 0, s, T, E, nblk, p_part, p_mean);
    return cudaGetLastError();
}

}  // namespace moe
