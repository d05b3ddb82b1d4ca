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
// probability p_i) and the histogram of the chosen ids (for the grouping scan).
//
// Two kernels:
//  * router_warp_kernel -- one warp per token, E <= 32 experts.  Each lane
//    streams 16-byte vectors of x and of the E rows of W_g (which stay hot in
//    L1 for small E*d), keeps E fp32 partial dots in registers and finishes
//    them with butterfly shuffles; afterwards lane e owns expert e.
//  * router_logits_kernel -- softmax/top-k over fp32 logits produced by a
//    tensor-core GEMM (large E); lane owns experts lane, lane+32, ...
#include <float.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = kRouterThreads / 32;
constexpr int kTokensPerWarp = kRouterTokensPerBlock / kWarps;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p + 4));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Softmax, top-k and gate epilogue shared by both kernels.  Lane L holds the
// logit (already including logit_bias) of experts L + 32*j in l[j]; absent
// experts hold -inf and index < 0.  Writes ids/gates for token t, adds p into
// the lane's running column sums and counts the chosen experts.
template <int NJ>
__device__ __forceinline__ void softmax_topk(int t, int E, int k, const float (&l)[NJ], const float* select_bias,
                                             int renormalize, int32_t* topk_ids, float* gates, float (&psum)[NJ],
                                             int (&hcnt)[NJ]) {
    const int lane = threadIdx.x & 31;
    float m = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < NJ; ++j)
        if (lane + 32 * j < E) m = fmaxf(m, l[j]);
    m = warp_max(m);
    float ex[NJ];
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        ex[j] = (lane + 32 * j < E) ? expf(l[j] - m) : 0.f;
        z += ex[j];
    }
    z = warp_sum(z);
    const float inv_z = 1.f / z;
    float p[NJ], s[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int e = lane + 32 * j;
        p[j] = ex[j] * inv_z;
        psum[j] += p[j];
        s[j] = (e < E) ? l[j] + (select_bias ? __ldg(select_bias + e) : 0.f) : -FLT_MAX;
    }
    uint32_t taken = 0;
    float gsum = 0.f;
    float my_gate = 0.f;  // lane r keeps the r-th choice (k <= 32)
    int my_id = -1;
    for (int r = 0; r < k; ++r) {
        float bv = -FLT_MAX;
        int bi = -1;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !(taken >> j & 1u) && (bi < 0 || s[j] > bv)) {
                bv = s[j];
                bi = e;
            }
        }
        warp_argmax(bv, bi);
        // the owner lane marks it taken and publishes its probability
        float pw = 0.f;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
            if (bi == lane + 32 * j) {
                taken |= 1u << j;
                pw = p[j];
                hcnt[j] += 1;
            }
        pw = __shfl_sync(0xffffffffu, pw, bi & 31);
        gsum += pw;
        if (lane == r) {
            my_gate = pw;
            my_id = bi;
        }
    }
    if (lane < k) {
        topk_ids[(size_t)t * k + lane] = my_id;
        gates[(size_t)t * k + lane] = renormalize ? my_gate / gsum : my_gate;
    }
}

// Writes the per-block partial sums of p and the per-block id histogram.
template <int NJ>
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
        for (int w = 0; w < kWarps; ++w) {  // fixed order: deterministic
            ps += s_p[w * E + e];
            hs += s_h[w * E + e];
        }
        if (p_part) p_part[(size_t)blockIdx.x * E + e] = ps;
        if (block_hist) block_hist[(size_t)blockIdx.x * E + e] = hs;
    }
}

template <typename T, int NE>
__global__ void __launch_bounds__(kRouterThreads) router_warp_kernel(
    int Tn, int d, int E, int k, const T* __restrict__ x, const T* __restrict__ wg,
    const float* __restrict__ logit_bias, const float* __restrict__ select_bias, int renormalize,
    int32_t* __restrict__ topk_ids, float* __restrict__ gates, float* __restrict__ p_part,
    int32_t* __restrict__ block_hist) {
    __shared__ float s_p[kWarps * NE];
    __shared__ int s_h[kWarps * NE];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float psum[1] = {0.f};
    int hcnt[1] = {0};
    for (int i = 0; i < kTokensPerWarp; ++i) {
        const int t = blockIdx.x * kRouterTokensPerBlock + warp * kTokensPerWarp + i;
        if (t >= Tn) break;  // warp-uniform
        const T* xr = x + (size_t)t * d;
        float acc[NE];
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[e] = 0.f;
#pragma unroll 2
        for (int c = lane * 8; c < d; c += 256) {
            float xv[8];
            load8(xr + c, xv);
#pragma unroll
            for (int e = 0; e < NE; ++e) {
                if (e < E) {
                    float wv[8];
                    load8(wg + (size_t)e * d + c, wv);
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[e] = fmaf(xv[q], wv[q], acc[e]);
                }
            }
        }
        float l[1] = {-FLT_MAX};
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            if (e < E) {
                const float v = warp_sum(acc[e]);
                if (lane == e) l[0] = v + (logit_bias ? __ldg(logit_bias + e) : 0.f);
            }
        }
        softmax_topk<1>(t, E, k, l, select_bias, renormalize, topk_ids, gates, psum, hcnt);
    }
    block_epilogue<1>(E, psum, hcnt, p_part, block_hist, s_p, s_h);
}

template <int NJ>
__global__ void __launch_bounds__(kRouterThreads) router_logits_kernel(
    int Tn, int E, int k, const float* __restrict__ logits, const float* __restrict__ logit_bias,
    const float* __restrict__ select_bias, int renormalize, int32_t* __restrict__ topk_ids,
    float* __restrict__ gates, float* __restrict__ p_part, int32_t* __restrict__ block_hist) {
    extern __shared__ float s_dyn[];
    float* s_p = s_dyn;
    int* s_h = reinterpret_cast<int*>(s_dyn + kWarps * E);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float psum[NJ];
    int hcnt[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        psum[j] = 0.f;
        hcnt[j] = 0;
    }
    for (int i = 0; i < kTokensPerWarp; ++i) {
        const int t = blockIdx.x * kRouterTokensPerBlock + warp * kTokensPerWarp + i;
        if (t >= Tn) break;
        float l[NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int e = lane + 32 * j;
            l[j] = (e < E) ? logits[(size_t)t * E + e] + (logit_bias ? __ldg(logit_bias + e) : 0.f) : -FLT_MAX;
        }
        softmax_topk<NJ>(t, E, k, l, select_bias, renormalize, topk_ids, gates, psum, hcnt);
    }
    block_epilogue<NJ>(E, psum, hcnt, p_part, block_hist, s_p, s_h);
}

__global__ void p_mean_kernel(int Tn, int E, int nblk, const float* __restrict__ p_part, float* __restrict__ p_mean) {
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
                               cudaStream_t s) {
    const int nblk = (T + kRouterTokensPerBlock - 1) / kRouterTokensPerBlock;
    if (nblk == 0) return cudaSuccess;
    const dim3 grid(nblk), block(kRouterThreads);
#define MOE_ROUTER_CASE(TY, NE)                                                                              \
    router_warp_kernel<TY, NE><<<grid, block, 0, s>>>(T, d, E, k, static_cast<const TY*>(x),                \
                                                      static_cast<const TY*>(w_gate), logit_bias, select_bias, \
                                                      renormalize, topk_ids, gates, p_part, block_hist)
    if (dtype == MOE_BF16) {
        if (E <= 8) MOE_ROUTER_CASE(__nv_bfloat16, 8);
        else if (E <= 16) MOE_ROUTER_CASE(__nv_bfloat16, 16);
        else MOE_ROUTER_CASE(__nv_bfloat16, 32);
    } else {
        if (E <= 8) MOE_ROUTER_CASE(float, 8);
        else if (E <= 16) MOE_ROUTER_CASE(float, 16);
        else MOE_ROUTER_CASE(float, 32);
    }
#undef MOE_ROUTER_CASE
    return cudaGetLastError();
}

cudaError_t launch_router_from_logits(int T, int E, int k, const float* logits, const float* logit_bias,
                                      const float* select_bias, int renormalize, int32_t* topk_ids,
                                      float* gates, float* p_part, int32_t* block_hist, cudaStream_t s) {
    const int nblk = (T + kRouterTokensPerBlock - 1) / kRouterTokensPerBlock;
    if (nblk == 0) return cudaSuccess;
    const size_t smem = (size_t)kWarps * E * (sizeof(float) + sizeof(int));
    const dim3 grid(nblk), block(kRouterThreads);
#define MOE_LOGITS_CASE(NJ)                                                                                  \
    do {                                                                                                     \
        cudaFuncSetAttribute(router_logits_kernel<NJ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        router_logits_kernel<NJ><<<grid, block, smem, s>>>(T, E, k, logits, logit_bias, select_bias,       \
                                                           renormalize, topk_ids, gates, p_part, block_hist); \
    } while (0)
    if (E <= 64) MOE_LOGITS_CASE(2);
    else if (E <= 256) MOE_LOGITS_CASE(8);
    else MOE_LOGITS_CASE(32);
#undef MOE_LOGITS_CASE
    return cudaGetLastError();
}

cudaError_t launch_p_mean(int T, int E, int nblk, const float* p_part, float* p_mean, cudaStream_t s) {
    p_mean_kernel<<<(E + 255) / 256, 256, 0, s>>>(T, E, nblk, p_part, p_mean);
    return cudaGetLastError();
}

}  // namespace moe
