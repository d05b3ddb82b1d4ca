// route_math.cuh -- the router's per-token arithmetic, shared by every kernel
// that routes tokens (router.cu; decode_fused.cu, which recomputes the
// routing of a small batch in each of its CTAs and must agree with the
// one-block-per-token router bit for bit).
//
// Per token t ("Mixture of Experts" notes, How it works: g(x) = softmax(W_g x),
// keep the top-k, renormalise; "Mixture of experts (MoE)" handbook, Load
// balancing: the per-expert bias steers the choice only):
//   p   = softmax(l),  l = W_g x_t + logit_bias
//   ids = top-k of l + select_bias, descending, ties to the lower index
//   g_j = p[ids_j] / sum_j p[ids_j]   (or p[ids_j] without renormalisation)
#pragma once

#include <float.h>

#include "common.cuh"

namespace moe {
namespace route_math {

// The one-block-per-token router (decode-sized batches) splits d over this
// many threads; its logits are sums in that thread order.
constexpr int kSplitDThreads = 512;

// 16-byte vector of T: 8 bf16 or 4 fp32.
template <typename T>
struct Vec {
    static constexpr int kElems = 16 / sizeof(T);
};

// acc += a.lo b.lo, then + a.hi b.hi: mixed-precision FMAs on bf16 operands
// into an fp32 accumulator.  A product of two bf16 values is exact in fp32,
// so each step rounds only the addition, as fmaf on the widened values would
// (the same result in one instruction, without widening either operand).
__device__ __forceinline__ float fma2_bf16(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

__device__ __forceinline__ void widen(const uint4& u, float (&v)[8], const __nv_bfloat16*) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ void widen(const uint4& u, float (&v)[4], const float*) {
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[3] = __uint_as_float(u.w);
}

// Softmax, top-k and gate epilogue of every router kernel.  Lane L holds the
// logit (already including logit_bias) of experts L + 32*j in l[j]; absent
// experts hold -inf and index < 0.  Writes ids/gates for token t, adds p into
// the lane's running column sums and counts the chosen experts.
template <int NJ>
__device__ __forceinline__ void softmax_topk(int t, int E, int k, const float (&l)[NJ], const float* select_bias,
                                             int renormalize, int32_t* topk_ids, float* gates, float (&psum)[NJ],
                                             int (&hcnt)[NJ], float* probs_out) {
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
        if (probs_out && e < E) probs_out[(size_t)t * E + e] = p[j];
        s[j] = (e < E) ? l[j] + (select_bias ? __ldg(select_bias + e) : 0.f) : -FLT_MAX;
        // a NaN score selects as -inf: the comparisons below then form a total
        // order (value, then lower index), so every lane agrees on each choice
        // and the ids match the histogram counted from them
        if (isnan(s[j])) s[j] = -INFINITY;
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

}  // namespace route_math
}  // namespace moe
