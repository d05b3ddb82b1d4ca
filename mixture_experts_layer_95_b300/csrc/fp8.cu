// fp8.cu -- FP8 (E4M3) quantisation of expert weights, one scale per row.
//
// The pages name FP8 quantisation of the experts as the way to fit them all
// in memory ("Mixture of Experts" notes, serving: INT4/FP8 "especially
// valuable"; handbook, DeepSeek-V3's FP8 weights) and warn that experts
// calibrate unevenly ("One Deep Concept #04" s13), but fix no scheme.  Here:
// OCP E4M3 codes with one fp32 scale per output channel, i.e. per row of
// every weight matrix (W1/W3 rows are the F hidden channels, W2 rows the d
// output channels):
//   scale = max_i |w_i| / 448   (1 for an all-zero row)
//   q_i   = E4M3(w_i / scale)   (IEEE fp32 quotient, round to nearest even,
//                                saturating at +-448)
// The expert GEMMs widen the codes exactly to bf16 and apply the scale to the
// fp32 accumulator of each output column.
//
// quantize_fp8_kernel: one warp per row, 16-byte loads; the row's maximum is
// a warp reduction, then the same warp re-reads the row (from L1/L2) and
// writes 8 codes per lane per step.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "fp8_split.cuh"

namespace moe {
namespace {

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}

template <typename T>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(long long rows, int cols, const T* __restrict__ w,
                                                           uint8_t* __restrict__ q, float* __restrict__ scale) {
    pdl_wait();
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row < rows) {
        const T* src = w + row * cols;
        float amax = 0.f;
        for (int c = lane * 8; c < cols; c += 256) {
            float v[8];
            load8<T>(src + c, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
        amax = warp_max(amax);
        const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        if (lane == 0) scale[row] = sc;
        uint8_t* dst = q + row * cols;
        for (int c = lane * 8; c < cols; c += 256) {
            float v[8];
            load8<T>(src + c, v);
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                lo |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(v[i], sc), __NV_SATFINITE, __NV_E4M3) << (8 * i);
                hi |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(v[4 + i], sc), __NV_SATFINITE, __NV_E4M3) << (8 * i);
            }
            *reinterpret_cast<uint2*>(dst + c) = make_uint2(lo, hi);
        }
    }
    __syncthreads();
    pdl_trigger();
}

// split_e4m3_kernel: one block per row of a bf16 matrix [rows][K] (K a
// multiple of 8) -> the E4M3 hi/lo code rows and power-of-two scale of
// fp8_split.cuh.  Row r of the output is row gather[r] of x when gather is
// given (token rows in expert order); rows at or beyond *live_rows (when
// given) are skipped.
constexpr int kSplitThreads = 256;

__global__ void __launch_bounds__(kSplitThreads) split_e4m3_kernel(int K, const __nv_bfloat16* __restrict__ x,
                                                                   int x_rows, const int32_t* __restrict__ gather,
                                                                   const int32_t* __restrict__ live_rows,
                                                                   uint8_t* __restrict__ hi, uint8_t* __restrict__ lo,
                                                                   float* __restrict__ scale) {
    __shared__ float s_max[kSplitThreads / 32];
    pdl_wait();
    const int row = blockIdx.x;
    int src_row = row;
    if (gather) {
        src_row = __ldg(gather + row);
        if (src_row < 0 || src_row >= x_rows) src_row = -1;  // the grouping scan wrote it; never taken
    }
    if ((!live_rows || row < __ldg(live_rows)) && src_row >= 0) {
        const __nv_bfloat16* src = x + (size_t)src_row * K;
        float amax = 0.f;
        for (int c = threadIdx.x * 8; c < K; c += kSplitThreads * 8) {
            float v[8];
            load8<__nv_bfloat16>(src + c, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
        amax = warp_max(amax);
        if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = amax;
        __syncthreads();
        amax = s_max[0];
#pragma unroll
        for (int w = 1; w < kSplitThreads / 32; ++w) amax = fmaxf(amax, s_max[w]);
        const E4m3RowScale sc = e4m3_row_scale(amax);
        if (threadIdx.x == 0) scale[row] = sc.s;
        uint8_t* dh = hi + (size_t)row * K;
        uint8_t* dl = lo + (size_t)row * K;
        for (int c = threadIdx.x * 8; c < K; c += kSplitThreads * 8) {
            float v[8];
            load8<__nv_bfloat16>(src + c, v);
            uint2 h, l;
            e4m3_split8(v, sc, h, l);
            *reinterpret_cast<uint2*>(dh + c) = h;
            *reinterpret_cast<uint2*>(dl + c) = l;
        }
    }
    __syncthreads();
    pdl_trigger();
}

}  // namespace

cudaError_t launch_split_e4m3(int rows, int K, const void* x, int x_rows, const int32_t* gather,
                              const int32_t* live_rows, uint8_t* hi, uint8_t* lo, float* scale, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    if (K % 8 != 0) return cudaErrorInvalidValue;
    launch_pdl(split_e4m3_kernel, dim3((unsigned)rows), dim3(kSplitThreads), 0, s, K,
               static_cast<const __nv_bfloat16*>(x), x_rows, gather, live_rows, hi, lo, scale);
    return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(int dtype, long long rows, int cols, const void* w, uint8_t* q, float* scale,
                                cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (dtype == MOE_BF16)
        launch_pdl(quantize_fp8_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0, s, rows, cols,
                   static_cast<const __nv_bfloat16*>(w), q, scale);
    else
        launch_pdl(quantize_fp8_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, s, rows, cols,
                   static_cast<const float*>(w), q, scale);
    return cudaGetLastError();
}

}  // namespace moe
