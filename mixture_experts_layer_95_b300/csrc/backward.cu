// backward.cu -- the transpose and router kernels of the backward
// pass; its matrix products run on the grouped tensor-core GEMM (gemm_tc.cu).
//
// Gradients of <dy, y> + dL * L_balance with the routing decisions held fixed
// (top-k selection has no gradient) and f_i held constant while p_i carries the
// gradient ("MoE Deep Dive", Load Balancing Loss Derivation).  Per kept slot
// (row r of the permuted layout, expert e, gate g), with G = X W1^T, U = X W3^T
// recomputed and D = dy W2_e (the down projection transposed; the GEMM reads
// W2_e, W1_e and W3_e as stored, as MN-major B operands):
//   dg_r = sum_f D h,   h = silu(G) U
//   dh = g D,  dG = dh U silu'(G),  dU = dh silu(G)
//   dX_r = dG W1_e + dU W3_e,  dW1_e = dG^T X,  dW3_e = dU^T X,  dW2_e = (g dy)^T h
// The element-wise part (h, dh, dG, dU, dg) runs in the epilogue of the D
// GEMM (kGemmSwigluBwd).  The weight gradients contract over each expert's
// token rows: their operands are transposed per expert into K windows that
// start on 64-column boundaries (zero-filled to the next boundary), which the
// GEMM's K-grouped mode reads.
#include "common.cuh"

namespace moe {
namespace {

constexpr int TT = 64;  // transpose tile

__device__ __forceinline__ float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }

// kbase[e] = sum over e' < e of klen rounded up to 64, klen[e] = rows of expert e.
// const_len >= 0: a single window of that many rows, and offsets (then an
// output) = {0, const_len}.
__global__ void k_windows_kernel(int E, int32_t* __restrict__ offsets, int32_t* __restrict__ kbase,
                                 int32_t* __restrict__ klen, int const_len) {
    pdl_wait();
    if (threadIdx.x == 0) {
        if (const_len >= 0) {
            offsets[0] = 0;
            offsets[1] = const_len;
            kbase[0] = 0;
            klen[0] = const_len;
        } else {
            int run = 0;
            for (int e = 0; e < E; ++e) {
                const int len = max(0, offsets[e + 1] - offsets[e]);
                kbase[e] = run;
                klen[e] = len;
                run += (len + 63) / 64 * 64;
            }
        }
    }
    __syncthreads();
    pdl_trigger();
}

// A block moves 64 window columns (source rows) x 128 source columns.  The
// tile is staged in shared memory as 32-bit words, word w of source column c
// holding rows 2w and 2w+1 (the bf16 pair that lands side by side in the
// destination row), so both phases move whole words: the load phase pairs
// two rows' 16-byte chunks with byte permutes, the store phase reads 16-byte
// runs of a column.  Word w of column c sits at w ^ tile_swizzle(c), which
// puts the 32 word stores of a load-phase warp on 32 banks and keeps each
// 16-byte run of the store phase in one 4-word group (its two halves swapped
// when bit 1 of the swizzle is set).  All of a thread's loads are issued
// before the first shared-memory store, so each SM keeps up to 128 KB of
// reads in flight.
constexpr int TC = 128;  // source columns per block
constexpr int TW = TT / 2;  // words per staged column

__device__ __forceinline__ int tile_swizzle(int c) {
    const int ch = c >> 3;  // the 8-column chunk of the source row
    return ((ch & 7) << 2) | ((ch >> 3) << 1);
}

// dst[c][kbase[e] + k] = scale(row) * src[(offsets[e] + k) * ld_src + col0 + c] for
// k < klen[e], 0 for klen[e] <= k < round64(klen[e]); c < C.  A block's 64
// destination columns lie inside one expert's window.  C, ld_src, col0 and
// ld_dst are multiples of 8 (16-byte chunks).
__global__ void __launch_bounds__(256, 8) transpose_windows_kernel(const __nv_bfloat16* __restrict__ src, size_t ld_src,
                                                                int col0, int C, int E,
                                                                const int32_t* __restrict__ offsets,
                                                                const int32_t* __restrict__ kbase,
                                                                const int32_t* __restrict__ klen,
                                                                const float* __restrict__ row_scale,
                                                                __nv_bfloat16* __restrict__ dst, size_t ld_dst,
                                                                int ncols) {
    pdl_wait();
    __shared__ __align__(16) uint32_t tile[TC * TW];
    const int c_tile = blockIdx.x * TC;  // source column block
    const int k0 = blockIdx.y * TT;      // destination column block
    if (k0 < ncols) {
        int lo = 0, hi = E - 1;  // last expert whose window starts at or before k0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(kbase + mid) <= k0) lo = mid;
            else hi = mid - 1;
        }
        const int e = lo;
        const int base = __ldg(kbase + e), len = __ldg(klen + e);
        const int padded = (len + 63) / 64 * 64;
        if (k0 < base + padded) {  // beyond the last window: nothing to write
            const int row_base = __ldg(offsets + e) + (k0 - base);
            // load: 32 row pairs x 16 chunks of 8 columns, two (pair, chunk) items per thread
            constexpr int kItems = (TW * (TC / 8)) / 256;
            uint4 v[kItems][2];
#pragma unroll
            for (int it = 0; it < kItems; ++it) {
                const int i = threadIdx.x + it * 256;
                const int ch = i & (TC / 8 - 1), p = i / (TC / 8);
                const int c = c_tile + ch * 8;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int kk = 2 * p + h;
                    v[it][h] = make_uint4(0u, 0u, 0u, 0u);
                    if (k0 - base + kk < len && c < C)
                        v[it][h] = __ldg(reinterpret_cast<const uint4*>(src + (size_t)(row_base + kk) * ld_src + col0 + c));
                }
            }
#pragma unroll
            for (int it = 0; it < kItems; ++it) {
                const int i = threadIdx.x + it * 256;
                const int ch = i & (TC / 8 - 1), p = i / (TC / 8);
                if (row_scale) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int kk = 2 * p + h;
                        if (k0 - base + kk >= len) continue;
                        const float sc = __ldg(row_scale + row_base + kk);
                        __nv_bfloat162* b = reinterpret_cast<__nv_bfloat162*>(&v[it][h]);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float2 f = __bfloat1622float2(b[j]);
                            b[j] = __floats2bfloat162_rn(f.x * sc, f.y * sc);
                        }
                    }
                }
                const uint32_t a[4] = {v[it][0].x, v[it][0].y, v[it][0].z, v[it][0].w};
                const uint32_t b[4] = {v[it][1].x, v[it][1].y, v[it][1].z, v[it][1].w};
                const int sw = tile_swizzle(ch * 8);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = ch * 8 + 2 * j;  // source columns c (low halves) and c + 1 (high halves)
                    tile[c * TW + (p ^ sw)] = __byte_perm(a[j], b[j], 0x5410);
                    tile[(c + 1) * TW + (p ^ sw)] = __byte_perm(a[j], b[j], 0x7632);
                }
            }
            __syncthreads();
            // store: 128 destination rows (source columns) x 8 runs of 8 window columns
#pragma unroll
            for (int it = 0; it < (TC * 8) / 256; ++it) {
                const int i = threadIdx.x + it * 256;
                const int cc = i >> 3, q = i & 7;
                if (c_tile + cc >= C) continue;
                const int sw = tile_swizzle(cc);
                uint4 w = *reinterpret_cast<const uint4*>(&tile[cc * TW + 4 * (q ^ (sw >> 2))]);
                if (sw & 2) w = make_uint4(w.z, w.w, w.x, w.y);
                *reinterpret_cast<uint4*>(dst + (size_t)(c_tile + cc) * ld_dst + k0 + q * 8) = w;
            }
        }
    }
    __syncthreads();
    pdl_trigger();
}

// Gates -> logits for token t (one warp per token), plus the balance loss:
//   renormalised gates:  dl[e_j] = g_j (dg_j - sum_j' g_j' dg_j')
//   plain gates (p):     dl = p (u - <p, u>), u[e_j] = dg_j
//   balance loss:        dl += dL alpha E / T  p (f - <p, f>),  f = counts / (T k)
__global__ void __launch_bounds__(256) router_backward_kernel(int Tn, int E, int k, const float* __restrict__ probs,
                                                              const int32_t* __restrict__ ids,
                                                              const int32_t* __restrict__ slot_pos,
                                                              const float* __restrict__ gates,
                                                              const float* __restrict__ dgp, int renormalize,
                                                              const int32_t* __restrict__ counts, float alpha,
                                                              float dL, float* __restrict__ dlogits) {
    pdl_wait();
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t < Tn) {
        const float* p = probs + (size_t)t * E;
        float* dl = dlogits + (size_t)t * E;
        // lane j < k: this token's slot j
        float dg = 0.f, gj = 0.f, pj = 0.f;
        int ej = -1;
        if (lane < k) {
            ej = __ldg(ids + (size_t)t * k + lane);
            const int pos = __ldg(slot_pos + (size_t)t * k + lane);
            dg = pos >= 0 ? __ldg(dgp + pos) : 0.f;
            gj = __ldg(gates + (size_t)t * k + lane);
            pj = (ej >= 0 && ej < E) ? __ldg(p + ej) : 0.f;
        }
        const float s = warp_sum(renormalize ? gj * dg : pj * dg);
        const float inv_tk = 1.0f / ((float)Tn * (float)k);
        float pf = 0.f;
        for (int e = lane; e < E; e += 32) pf += __ldg(p + e) * ((float)__ldg(counts + e) * inv_tk);
        pf = warp_sum(pf);
        const float c = dL * alpha * (float)E / (float)Tn;
        for (int e = lane; e < E; e += 32) {
            const float pe = __ldg(p + e);
            float v = c * pe * ((float)__ldg(counts + e) * inv_tk - pf);
            if (!renormalize) v -= pe * s;
            dl[e] = v;
        }
        __syncwarp();
        if (lane < k && ej >= 0 && ej < E) dl[ej] += renormalize ? gj * (dg - s) : pj * dg;
    }
    __syncthreads();
    pdl_trigger();
}

// R[t][i] = sum_e dl[t][e] W_g[e][i] (+ extra[t][i]): 8 tokens x 256 columns per block.
template <typename T>
__global__ void __launch_bounds__(256) router_dx_kernel(int Tn, int E, int d, const float* __restrict__ dlogits,
                                                        const T* __restrict__ wg, const float* __restrict__ extra,
                                                        float* __restrict__ R) {
    pdl_wait();
    constexpr int TOK = 8;
    __shared__ float s_dl[TOK][128];
    const int t0 = blockIdx.y * TOK;
    const int i = blockIdx.x * 256 + threadIdx.x;
    float acc[TOK];
#pragma unroll
    for (int q = 0; q < TOK; ++q) acc[q] = 0.f;
    for (int e0 = 0; e0 < E; e0 += 128) {
        __syncthreads();
        for (int j = threadIdx.x; j < TOK * 128; j += blockDim.x) {
            const int q = j / 128, e = e0 + j % 128;
            s_dl[q][j % 128] = (t0 + q < Tn && e < E) ? __ldg(dlogits + (size_t)(t0 + q) * E + e) : 0.f;
        }
        __syncthreads();
        if (i < d) {
            const int ne = min(128, E - e0);
            for (int e = 0; e < ne; ++e) {
                float w;
                if constexpr (sizeof(T) == 2) w = bf2f(wg[(size_t)(e0 + e) * d + i]);
                else w = wg[(size_t)(e0 + e) * d + i];
#pragma unroll
                for (int q = 0; q < TOK; ++q) acc[q] = fmaf(s_dl[q][e], w, acc[q]);
            }
        }
    }
    if (i < d)
#pragma unroll
        for (int q = 0; q < TOK; ++q)
            if (t0 + q < Tn)
                R[(size_t)(t0 + q) * d + i] = acc[q] + (extra ? __ldg(extra + (size_t)(t0 + q) * d + i) : 0.f);
    __syncthreads();
    pdl_trigger();
}

// part[s][e][i] = sum over tokens t of chunk s of dl[t][e] x[t][i]: EB experts x
// 512 columns per block (two adjacent columns per thread), the tokens split into
// `nsplit` chunks (summed afterwards in chunk order).  Each thread loads the x
// values of 32 tokens before it multiplies any of them, so the loads of a batch
// are in flight together; within a chunk the tokens are added in index order.
template <typename T, int EB>
__global__ void __launch_bounds__(256) wgate_grad_kernel(int Tn, int E, int d, const float* __restrict__ dlogits,
                                                         const T* __restrict__ x, int nsplit,
                                                         float* __restrict__ part) {
    pdl_wait();
    constexpr int TB = 32;
    __shared__ float s_dl[TB][EB];
    const int e0 = blockIdx.y * EB;
    const int i = (blockIdx.x * 256 + threadIdx.x) * 2;  // columns i and i + 1 (d is even)
    const int s = blockIdx.z;
    const int tchunk = (Tn + nsplit - 1) / nsplit;
    const int ta = min(Tn, s * tchunk), tb = min(Tn, ta + tchunk);
    float acc0[EB], acc1[EB];
#pragma unroll
    for (int q = 0; q < EB; ++q) acc0[q] = acc1[q] = 0.f;
    for (int tt = ta; tt < tb; tt += TB) {
        __syncthreads();
        for (int j = threadIdx.x; j < TB * EB; j += blockDim.x) {
            const int q = j / EB, e = e0 + j % EB;
            s_dl[q][j % EB] = (tt + q < tb && e < E) ? __ldg(dlogits + (size_t)(tt + q) * E + e) : 0.f;
        }
        __syncthreads();
        if (i < d) {
            float x0[TB], x1[TB];
#pragma unroll
            for (int q = 0; q < TB; ++q) {
                x0[q] = x1[q] = 0.f;
                if (tt + q < tb) {
                    const size_t at = (size_t)(tt + q) * d + i;
                    if constexpr (sizeof(T) == 2) {
                        const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + at));
                        x0[q] = v.x;
                        x1[q] = v.y;
                    } else {
                        const float2 v = *reinterpret_cast<const float2*>(x + at);
                        x0[q] = v.x;
                        x1[q] = v.y;
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < TB; ++q)
#pragma unroll
                for (int e = 0; e < EB; ++e) {
                    acc0[e] = fmaf(s_dl[q][e], x0[q], acc0[e]);
                    acc1[e] = fmaf(s_dl[q][e], x1[q], acc1[e]);
                }
        }
    }
    if (i < d)
#pragma unroll
        for (int e = 0; e < EB; ++e)
            if (e0 + e < E)
                *reinterpret_cast<float2*>(part + ((size_t)s * E + e0 + e) * d + i) = make_float2(acc0[e], acc1[e]);
    __syncthreads();
    pdl_trigger();
}

int wgate_expert_block(int E) { return E <= 8 ? 8 : (E <= 16 ? 16 : 32); }

template <typename T, int EB>
void launch_wgate_eb(dim3 grid, cudaStream_t s, int T_, int E, int d, const float* dlogits, const void* x, int nsplit,
                     float* part) {
    launch_pdl(wgate_grad_kernel<T, EB>, grid, dim3(256), 0, s, T_, E, d, dlogits, static_cast<const T*>(x), nsplit,
               part);
}

template <typename T>
void launch_wgate_t(dim3 grid, cudaStream_t s, int T_, int E, int d, const float* dlogits, const void* x, int nsplit,
                    float* part) {
    switch (wgate_expert_block(E)) {
        case 8: launch_wgate_eb<T, 8>(grid, s, T_, E, d, dlogits, x, nsplit, part); break;
        case 16: launch_wgate_eb<T, 16>(grid, s, T_, E, d, dlogits, x, nsplit, part); break;
        default: launch_wgate_eb<T, 32>(grid, s, T_, E, d, dlogits, x, nsplit, part); break;
    }
}

}  // namespace

cudaError_t launch_k_windows(int E, int32_t* offsets, int32_t* kbase, int32_t* klen, int const_len, cudaStream_t s) {
    launch_pdl(k_windows_kernel, dim3(1), dim3(32), 0, s, E, offsets, kbase, klen, const_len);
    return cudaGetLastError();
}

cudaError_t launch_transpose_windows(const void* src, size_t ld_src, int col0, int C, int E, const int32_t* offsets,
                                     const int32_t* kbase, const int32_t* klen, const float* row_scale, void* dst,
                                     size_t ld_dst, int ncols, cudaStream_t s) {
    if (C == 0 || ncols == 0) return cudaSuccess;
    if (C % 8 || ld_src % 8 || col0 % 8 || ld_dst % 8 || ncols % 64) return cudaErrorInvalidValue;
    const dim3 grid((C + TC - 1) / TC, (ncols + TT - 1) / TT);
    launch_pdl(transpose_windows_kernel, grid, dim3(256), 0, s, static_cast<const __nv_bfloat16*>(src), ld_src, col0,
               C, E, offsets, kbase, klen, row_scale, static_cast<__nv_bfloat16*>(dst), ld_dst, ncols);
    return cudaGetLastError();
}

cudaError_t launch_router_backward(int T, int E, int k, const float* probs, const int32_t* ids,
                                   const int32_t* slot_pos, const float* gates, const float* dgp, int renormalize,
                                   const int32_t* counts, float alpha, float dL, float* dlogits, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    launch_pdl(router_backward_kernel, dim3((T + 7) / 8), dim3(256), 0, s, T, E, k, probs, ids, slot_pos, gates, dgp,
               renormalize, counts, alpha, dL, dlogits);
    return cudaGetLastError();
}

cudaError_t launch_router_dx(int dtype, int T, int E, int d, const float* dlogits, const void* w_gate,
                             const float* extra, float* R, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((d + 255) / 256, (T + 7) / 8);
    if (dtype == MOE_BF16)
        launch_pdl(router_dx_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, T, E, d, dlogits,
                   static_cast<const __nv_bfloat16*>(w_gate), extra, R);
    else
        launch_pdl(router_dx_kernel<float>, grid, dim3(256), 0, s, T, E, d, dlogits,
                   static_cast<const float*>(w_gate), extra, R);
    return cudaGetLastError();
}

int wgate_grad_split(int E, int d) {
    // about two waves of blocks on 148 SMs, at most 32 token chunks
    const long long blocks = (long long)((d + 511) / 512) * ((E + wgate_expert_block(E) - 1) / wgate_expert_block(E));
    long long sp = (2LL * 148 + blocks - 1) / blocks;
    return (int)(sp < 1 ? 1 : (sp > 32 ? 32 : sp));
}

cudaError_t launch_wgate_grad(int dtype, int T, int E, int d, const float* dlogits, const void* x, int nsplit,
                              float* part, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (d % 2 || nsplit < 1) return cudaErrorInvalidValue;
    const int eb = wgate_expert_block(E);
    const dim3 grid((d + 511) / 512, (E + eb - 1) / eb, nsplit);
    if (dtype == MOE_BF16)
        launch_wgate_t<__nv_bfloat16>(grid, s, T, E, d, dlogits, x, nsplit, part);
    else
        launch_wgate_t<float>(grid, s, T, E, d, dlogits, x, nsplit, part);
    return cudaGetLastError();
}

}  // namespace moe
