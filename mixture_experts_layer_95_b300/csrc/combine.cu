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
// Selection-bias update of auxiliary-loss-free balancing ("MoE Architecture"
// s2: over-loaded experts get a negative bias; handbook Load balancing: an
// overloaded expert's bias is lowered and an idle one's raised):
//   b_e -= gamma * sign(counts_e - T k / E), compared exactly in integers.
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

// 8 consecutive values of a row (16-byte aligned) as two float4: fp32 rows,
// or bf16 rows widened exactly
__device__ __forceinline__ void load8(const float* p, float4& a, float4& b) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p) + 1);
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float4& a, float4& b) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.z));
    const float2 f3 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.w));
    a = make_float4(f0.x, f0.y, f1.x, f1.y);
    b = make_float4(f2.x, f2.y, f3.x, f3.y);
}

// v rounded to bf16 and back (what storing it as a bf16 row would keep)
__device__ __forceinline__ float4 round_bf16(float4 v) {
    const float2 a = __bfloat1622float2(__floats2bfloat162_rn(v.x, v.y));
    const float2 b = __bfloat1622float2(__floats2bfloat162_rn(v.z, v.w));
    return make_float4(a.x, a.y, b.x, b.y);
}

// One warp per (token, CH 256-column chunks), so that even a single token is
// spread over d/(256 CH) warps.  The warp reads the token's k slot positions
// 32 at a time (lane j holds slot j of the batch), finds the live ones (>= 0)
// with a ballot and takes them NB at a time in ascending slot order, so that
// those rows' loads for every chunk are in flight together; each lane owns 8
// consecutive columns of each chunk.  Measured (same box, A/B): CH = 2,
// NB = 2 for k <= 2 without split-K slices (skewed layer 43 -> 32 us,
// Mixtral prefill 48 -> 36 us); one chunk and one row at a time otherwise,
// where the larger shapes cost more in warps per SM than they gain
// (DeepSeek-V3 shape, k = 8: 0.34 -> 0.36 ms; 128 decode tokens with slices:
// 15 -> 21 us).  k is the top-k of
// token choice, or E for expert choice (slot e live iff expert e took the
// token; n_empty, when given, counts the tokens with no live slot).  Rows of
// y_perm (and y_shared) may be split into `nsplit` fp32 slices `stride`
// elements apart: each entry's slices are summed in slice order first, then
// the entries in ascending j order, then the shared row -- the same order in
// which a reduction of the slices followed by the plain combine adds them.
// TIN: the rows' storage (fp32, or bf16 for layers that keep them in bf16).
// round_rows (fp32 split-K slices of a layer whose rows are bf16): each
// entry's slice sum is rounded to bf16 before it is added, exactly as if the
// slices had been reduced into a bf16 row first.

// One entry's 8 columns at c of row `pos`: its slices summed in slice order,
// rounded to bf16 when the layer keeps its rows in bf16.
template <bool SPLIT, typename TIN>
__device__ __forceinline__ void entry8(const TIN* __restrict__ rows, size_t stride, int nsplit, size_t pos, int d,
                                       int c, int round_rows, float4& p0, float4& p1) {
    load8(rows + pos * d + c, p0, p1);
    if (!SPLIT) return;
#pragma unroll 8
    for (int sl = 1; sl < nsplit; ++sl) {  // independent loads: keep them in flight together
        float4 q0, q1;
        load8(rows + sl * stride + pos * d + c, q0, q1);
        add4(p0, q0);
        add4(p1, q1);
    }
    if (round_rows) {
        p0 = round_bf16(p0);
        p1 = round_bf16(p1);
    }
}

template <typename T, typename TIN, int CH, int NB, bool SPLIT>
__global__ void __launch_bounds__(256) combine_kernel(int Tn, int d, int k, const TIN* __restrict__ y_perm,
                                                      size_t perm_stride, int nsplit,
                                                      const int32_t* __restrict__ slot_pos,
                                                      const TIN* __restrict__ y_shared, size_t shared_stride,
                                                      int shared_nsplit, T* __restrict__ y,
                                                      int32_t* __restrict__ n_empty, int round_rows) {
    pdl_wait();
    const int chunks = (d + 255) / 256;
    const int groups = (chunks + CH - 1) / CH;
    const int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (item >= Tn * groups) return;
    const int t = item / groups;
    const int g0 = (item - t * groups) * CH;
    int c[CH];
    bool act[CH];  // d is a multiple of 8: an active lane owns 8 columns of the chunk
#pragma unroll
    for (int h = 0; h < CH; ++h) {
        c[h] = (g0 + h) * 256 + lane * 8;
        act[h] = c[h] < d;
    }
    float4 acc[CH][2];
#pragma unroll
    for (int h = 0; h < CH; ++h) acc[h][0] = acc[h][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    bool any = false;
    for (int j0 = 0; j0 < k; j0 += 32) {  // 32 slots at a time; live ones in ascending j
        const int my_pos = j0 + lane < k ? __ldg(slot_pos + (size_t)t * k + j0 + lane) : -1;
        unsigned live = __ballot_sync(0xffffffffu, my_pos >= 0);
        any |= live != 0u;
        while (live) {  // warp-uniform
            int pos[NB];
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                pos[u] = -1;
                if (live) {
                    pos[u] = __shfl_sync(0xffffffffu, my_pos, __ffs(live) - 1);
                    live &= live - 1u;
                }
            }
            float4 q[NB][CH][2];
#pragma unroll
            for (int u = 0; u < NB; ++u)
#pragma unroll
                for (int h = 0; h < CH; ++h)
                    if (act[h] && pos[u] >= 0)
                        entry8<SPLIT>(y_perm, perm_stride, nsplit, (size_t)pos[u], d, c[h], round_rows, q[u][h][0],
                                      q[u][h][1]);
#pragma unroll
            for (int u = 0; u < NB; ++u)
#pragma unroll
                for (int h = 0; h < CH; ++h)
                    if (act[h] && pos[u] >= 0) {
                        add4(acc[h][0], q[u][h][0]);
                        add4(acc[h][1], q[u][h][1]);
                    }
        }
    }
    if (n_empty && !any && lane == 0 && g0 == 0) atomicAdd(n_empty, 1);  // a token no expert took
#pragma unroll
    for (int h = 0; h < CH; ++h) {
        if (!act[h]) continue;
        if (y_shared) {
            float4 p0, p1;
            entry8<SPLIT>(y_shared, shared_stride, shared_nsplit, (size_t)t, d, c[h], round_rows, p0, p1);
            add4(acc[h][0], p0);
            add4(acc[h][1], p1);
        }
        store4<T>(y + (size_t)t * d + c[h], acc[h][0]);
        store4<T>(y + (size_t)t * d + c[h] + 4, acc[h][1]);
    }
}

// SwiGLU over split-K partials of the up GEMM: one thread per 4 columns.
__global__ void __launch_bounds__(256) swiglu_finalize_kernel(int rows_max, const int32_t* __restrict__ rows_dev,
                                                              int N, int ksplit, const float* __restrict__ part,
                                                              __nv_bfloat16* __restrict__ h,
                                                              __nv_bfloat16* __restrict__ h_lo) {
    pdl_wait();
    const int rows = rows_dev ? min(*rows_dev, rows_max) : rows_max;
    const size_t stride = (size_t)rows_max * 2 * N;
    const int q4 = N / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)rows * q4;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / q4;
        const int f = (int)(i - r * q4) * 4;
        const float* gp = part + r * 2 * N + f;
        float4 g = __ldg(reinterpret_cast<const float4*>(gp));
        float4 u = __ldg(reinterpret_cast<const float4*>(gp + N));
#pragma unroll 8
        for (int sl = 1; sl < ksplit; ++sl) {
            add4(g, __ldg(reinterpret_cast<const float4*>(gp + sl * stride)));
            add4(u, __ldg(reinterpret_cast<const float4*>(gp + sl * stride + N)));
        }
        const float hv[4] = {g.x / (1.0f + __expf(-g.x)) * u.x, g.y / (1.0f + __expf(-g.y)) * u.y,
                             g.z / (1.0f + __expf(-g.z)) * u.z, g.w / (1.0f + __expf(-g.w)) * u.w};
        __nv_bfloat162 a = __floats2bfloat162_rn(hv[0], hv[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(hv[2], hv[3]);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&a);
        pk.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(h + r * N + f) = pk;
        if (h_lo) {
            const float2 ba = __bfloat1622float2(a), bb = __bfloat1622float2(b);
            __nv_bfloat162 la = __floats2bfloat162_rn(hv[0] - ba.x, hv[1] - ba.y);
            __nv_bfloat162 lb = __floats2bfloat162_rn(hv[2] - bb.x, hv[3] - bb.y);
            pk.x = *reinterpret_cast<uint32_t*>(&la);
            pk.y = *reinterpret_cast<uint32_t*>(&lb);
            *reinterpret_cast<uint2*>(h_lo + r * N + f) = pk;
        }
    }
    __syncthreads();
    pdl_trigger();
}

// out[r][c] = sum over slices of part[s][r][c], slices in order (stored as
// fp32, or rounded to bf16).
template <typename TO>
__global__ void __launch_bounds__(256) reduce_partials_kernel(int rows_max, const int32_t* __restrict__ rows_dev,
                                                              int N, int ksplit, const float* __restrict__ part,
                                                              TO* __restrict__ out) {
    pdl_wait();
    const int rows = rows_dev ? min(*rows_dev, rows_max) : rows_max;
    const size_t stride = (size_t)rows_max * N;
    const int q4 = N / 4;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)rows * q4;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / q4;
        const int c = (int)(i - r * q4) * 4;
        float4 acc = __ldg(reinterpret_cast<const float4*>(part + r * N + c));
#pragma unroll 8
        for (int sl = 1; sl < ksplit; ++sl)
            add4(acc, __ldg(reinterpret_cast<const float4*>(part + sl * stride + r * N + c)));
        store4<TO>(out + r * N + c, acc);
    }
    __syncthreads();
    pdl_trigger();
}

int grid_for(size_t work, int per_block) {
    const size_t b = (work + per_block - 1) / per_block;
    return (int)(b < 148 * 16 ? (b > 0 ? b : 1) : 148 * 16);
}

__global__ void load_stats_kernel(int Tn, int E, int k, float alpha, const int32_t* __restrict__ counts,
                                  const float* __restrict__ p_mean, float* __restrict__ f, float* __restrict__ L) {
    pdl_wait();
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

__global__ void bias_update_kernel(int Tn, int E, int k, const int32_t* __restrict__ counts, float gamma,
                                   float* __restrict__ bias) {
    pdl_wait();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const long long scaled = (long long)counts[e] * E, total = (long long)Tn * k;
    if (scaled > total) bias[e] = bias[e] - gamma;
    else if (scaled < total) bias[e] = bias[e] + gamma;
}

}  // namespace

cudaError_t launch_bias_update(int T, int E, int k, const int32_t* counts, float gamma, float* bias, cudaStream_t s) {
    launch_pdl(bias_update_kernel, dim3((E + 255) / 256), dim3(256), 0, s, T, E, k, counts, gamma, bias);
    return cudaGetLastError();
}

template <typename T, typename TIN>
void launch_combine_kernel(int T_, int d, int k, const TIN* y_perm, size_t perm_stride, int nsplit,
                           const int32_t* slot_pos, const TIN* y_shared, size_t shared_stride, int shared_nsplit,
                           T* y, int32_t* n_empty, int round_rows, cudaStream_t s) {
    const int chunks = (d + 255) / 256;
    const bool split = nsplit > 1 || shared_nsplit > 1 || round_rows;
    const long long w2 = (long long)T_ * ((chunks + 1) / 2), w1 = (long long)T_ * chunks;
#define MOE_COMBINE(CH, NB, SP, W)                                                                              \
    launch_pdl(combine_kernel<T, TIN, CH, NB, SP>, dim3((int)(((W) + 7) / 8)), dim3(256), 0, s, T_, d, k, y_perm, \
               perm_stride, nsplit, slot_pos, y_shared, shared_stride, shared_nsplit, y, n_empty, round_rows)
    if (k <= 2 && !split) MOE_COMBINE(2, 2, false, w2);
    else if (split) MOE_COMBINE(1, 1, true, w1);
    else MOE_COMBINE(1, 1, false, w1);
#undef MOE_COMBINE
}

cudaError_t launch_combine_split(int dtype, int T, int d, int k, const float* y_perm, size_t perm_stride,
                                 int nsplit, const int32_t* slot_pos, const float* y_shared, size_t shared_stride,
                                 int shared_nsplit, void* y, cudaStream_t s, int32_t* n_empty, bool round_rows) {
    if (T == 0) return cudaSuccess;
    const int rr = round_rows ? 1 : 0;
    if (dtype == MOE_BF16)
        launch_combine_kernel(T, d, k, y_perm, perm_stride, nsplit, slot_pos, y_shared, shared_stride, shared_nsplit,
                              static_cast<__nv_bfloat16*>(y), n_empty, rr, s);
    else
        launch_combine_kernel(T, d, k, y_perm, perm_stride, nsplit, slot_pos, y_shared, shared_stride, shared_nsplit,
                              static_cast<float*>(y), n_empty, rr, s);
    return cudaGetLastError();
}

cudaError_t launch_combine(int dtype, int T, int d, int k, const void* y_perm, const int32_t* slot_pos,
                           const void* y_shared, void* y, cudaStream_t s, int32_t* n_empty, bool rows_bf16) {
    if (T == 0) return cudaSuccess;
    if (!rows_bf16)
        return launch_combine_split(dtype, T, d, k, static_cast<const float*>(y_perm), 0, 1, slot_pos,
                                    static_cast<const float*>(y_shared), 0, 1, y, s, n_empty, false);
    const __nv_bfloat16* yp = static_cast<const __nv_bfloat16*>(y_perm);
    const __nv_bfloat16* ys = static_cast<const __nv_bfloat16*>(y_shared);
    if (dtype == MOE_BF16)
        launch_combine_kernel(T, d, k, yp, (size_t)0, 1, slot_pos, ys, (size_t)0, 1, static_cast<__nv_bfloat16*>(y),
                              n_empty, 0, s);
    else
        launch_combine_kernel(T, d, k, yp, (size_t)0, 1, slot_pos, ys, (size_t)0, 1, static_cast<float*>(y), n_empty,
                              0, s);
    return cudaGetLastError();
}

cudaError_t launch_swiglu_finalize(int rows_max, const int32_t* rows_dev, int N, int ksplit, const float* part,
                                   void* h, void* h_lo, cudaStream_t s) {
    if (rows_max == 0) return cudaSuccess;
    launch_pdl(swiglu_finalize_kernel, dim3(grid_for((size_t)rows_max * (N / 4), 256)), dim3(256), 0, s, 
        rows_max, rows_dev, N, ksplit, part, static_cast<__nv_bfloat16*>(h), static_cast<__nv_bfloat16*>(h_lo));
    return cudaGetLastError();
}

cudaError_t launch_reduce_partials(int rows_max, const int32_t* rows_dev, int N, int ksplit, const float* part,
                                   void* out, cudaStream_t s, bool out_bf16) {
    if (rows_max == 0) return cudaSuccess;
    const dim3 grid(grid_for((size_t)rows_max * (N / 4), 256));
    if (out_bf16)
        launch_pdl(reduce_partials_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, rows_max, rows_dev, N, ksplit, part,
                   static_cast<__nv_bfloat16*>(out));
    else
        launch_pdl(reduce_partials_kernel<float>, grid, dim3(256), 0, s, rows_max, rows_dev, N, ksplit, part,
                   static_cast<float*>(out));
    return cudaGetLastError();
}

cudaError_t launch_load_stats(int T, int E, int k, float alpha, const int32_t* counts, const float* p_mean,
                              float* f, float* L, cudaStream_t s) {
    launch_pdl(load_stats_kernel, dim3(1), dim3(256), 0, s, T, E, k, alpha, counts, p_mean, f, L);
    return cudaGetLastError();
}

}  // namespace moe
