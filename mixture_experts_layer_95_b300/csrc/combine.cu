// combine.cu -- gate-weighted combine back to token order, and load statistics.
//
// Combine ("Mixture of experts (MoE)" handbook, forward_grouped: add each
// expert's weighted rows back at their tokens' positions, then add the shared
// expert; "MoE Architecture" s1, y = sum_i g_i Expert_i(x), and s3, shared
// experts process every token): the gate is already applied by the down-GEMM
// epilogue, so
//   y[t] = sum_{j : slot_pos[t][j] >= 0} y_perm[slot_pos[t][j]] + y_shared[t]
// summed in fixed j order in fp32 (deterministic, no atomics), one warp per
// token, 16-byte vector gathers.
//
// Load statistics ("MoE Architecture" s2 Load Balancing; handbook aux_loss):
//   f_i = counts_i / (T k),   L = alpha * E * sum_i f_i p_i.
#include "common.cuh"

namespace moe {
namespace {

template <typename T>
__device__ __forceinline__ void store4(T* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ void add4(float4& a, const float4& b) {
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// One warp per token.  Lane j < k holds slot_pos[t][j] (k <= 32) and
// broadcasts it; every lane then sums 8 consecutive columns per step (two
// 16-byte loads per row, all rows' loads issued before the adds) in the
// fixed order j = 0..k-1, then the shared row.
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(int Tn, int d, int k, const float* __restrict__ y_perm,
                                                      const int32_t* __restrict__ slot_pos,
                                                      const float* __restrict__ y_shared, T* __restrict__ y) {
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= Tn) return;
    const int my_pos = lane < k ? __ldg(slot_pos + (size_t)t * k + lane) : -1;
    // the loop bound is the same for every lane, so the shuffles below always
    // run with the whole warp; lanes past the row end skip only the memory work
    for (int c0 = 0; c0 < d; c0 += 256) {
        const int c = c0 + lane * 8;
        const bool active = c < d;  // d is a multiple of 8: an active lane owns 8 columns
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
        for (int j = 0; j < k; ++j) {
            const int pos = __shfl_sync(0xffffffffu, my_pos, j);
            if (pos < 0 || !active) continue;
            const float4* src = reinterpret_cast<const float4*>(y_perm + (size_t)pos * d + c);
            add4(a0, __ldg(src));
            add4(a1, __ldg(src + 1));
        }
        if (!active) continue;
        if (y_shared) {
            const float4* src = reinterpret_cast<const float4*>(y_shared + (size_t)t * d + c);
            add4(a0, __ldg(src));
            add4(a1, __ldg(src + 1));
        }
        store4<T>(y + (size_t)t * d + c, a0);
        store4<T>(y + (size_t)t * d + c + 4, a1);
    }
}

__global__ void load_stats_kernel(int Tn, int E, int k, float alpha, const int32_t* __restrict__ counts,
                                  const float* __restrict__ p_mean, float* __restrict__ f, float* __restrict__ L) {
    __shared__ float s_red[256];
    float part = 0.f;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const float fe = (float)counts[e] / ((float)Tn * (float)k);
        if (f) f[e] = fe;
        part += fe * p_mean[e];
    }
    s_red[threadIdx.x] = part;
    __syncthreads();
    if (threadIdx.x == 0 && L) {
        float acc = 0.f;
        for (int i = 0; i < (int)blockDim.x; ++i) acc += s_red[i];
        *L = alpha * (float)E * acc;
    }
}

}  // namespace

cudaError_t launch_combine(int dtype, int T, int d, int k, const float* y_perm, const int32_t* slot_pos,
                           const float* y_shared, void* y, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int grid = (T + 7) / 8;
    if (dtype == MOE_BF16)
        combine_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(T, d, k, y_perm, slot_pos, y_shared,
                                                           static_cast<__nv_bfloat16*>(y));
    else
        combine_kernel<float><<<grid, 256, 0, s>>>(T, d, k, y_perm, slot_pos, y_shared, static_cast<float*>(y));
    return cudaGetLastError();
}

cudaError_t launch_load_stats(int T, int E, int k, float alpha, const int32_t* counts, const float* p_mean,
                              float* f, float* L, cudaStream_t s) {
    load_stats_kernel<<<1, 256, 0, s>>>(T, E, k, alpha, counts, p_mean, f, L);
    return cudaGetLastError();
}

}  // namespace moe
