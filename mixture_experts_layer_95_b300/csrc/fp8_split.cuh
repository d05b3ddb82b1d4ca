// fp8_split.cuh -- the E4M3 hi/lo split of a bf16 row (device helpers).
//
// The FP8 tensor-core MMA (kind::f8f6f4) takes FP8 on both operands, so a
// bf16 row x that meets FP8 weights is carried as two E4M3 code rows and a
// power-of-two scale,  x = s * (hi + lo):
//   s  = 2^(e - 8) with max|x| = m * 2^e, m in [0.5, 1)  (1 for a zero row),
//        so |x| / s < 256 and the division by s is exact;
//   hi = E4M3(x / s), lo = E4M3(x / s - hi), both rounded to nearest even.
// hi keeps the top 4 significant bits of x / s and the remainder has at most
// 4 more (a bf16 value has 8), so hi + lo == x / s exactly whenever lo stays
// at or above E4M3's smallest step 2^-9, i.e. for every |x| >= max|x| * 2^-10;
// smaller entries carry an absolute error of at most s * 2^-10 <= max|x| *
// 2^-17.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

// 1/s as two factors (each inside the fp32 range) and s itself.
struct E4m3RowScale {
    float f1, f2, s;
};

__device__ __forceinline__ E4m3RowScale e4m3_row_scale(float amax) {
    int e = 8;  // zero row: s = 1
    if (amax > 0.f) frexpf(amax, &e);
    const int sh = 8 - e, sh1 = sh / 2, sh2 = sh - sh1;
    E4m3RowScale r;
    r.f1 = ldexpf(1.0f, sh1);
    r.f2 = ldexpf(1.0f, sh2);
    r.s = ldexpf(1.0f, e - 8);
    return r;
}

// 8 consecutive row entries -> 8 hi codes and 8 lo codes (element i in byte i).
__device__ __forceinline__ void e4m3_split8(const float (&v)[8], const E4m3RowScale& sc, uint2& hi, uint2& lo) {
    uint32_t h[2] = {0u, 0u}, l[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const float2 a = make_float2(v[i] * sc.f1 * sc.f2, v[i + 1] * sc.f1 * sc.f2);
        const __nv_fp8x2_storage_t hc = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hc, __NV_E4M3);
        const float2 hv = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        const float2 r = make_float2(a.x - hv.x, a.y - hv.y);
        const __nv_fp8x2_storage_t lc = __nv_cvt_float2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3);
        h[i >> 2] |= (uint32_t)hc << (16 * ((i >> 1) & 1));
        l[i >> 2] |= (uint32_t)lc << (16 * ((i >> 1) & 1));
    }
    hi = make_uint2(h[0], h[1]);
    lo = make_uint2(l[0], l[1]);
}

}  // namespace moe
