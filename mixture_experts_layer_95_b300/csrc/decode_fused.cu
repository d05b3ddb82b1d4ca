// decode_fused.cu -- the whole token-choice layer for one-token batches
// (kFusedMaxT) on routers of at most kFusedMaxE experts, in two launches.
//
// What it computes is what every other path of moe_forward computes (sources
// by page title and section): router logits, softmax, top-k and gates
// ("Mixture of Experts" notes, How it works), the capacity cut (same notes,
// capacity and token dropping), the SwiGLU expert down(silu(gate(x)) * up(x))
// ("Mixture of experts (MoE)" handbook, Structure), the gated sum of a token's
// expert outputs (handbook forward_naive), the shared expert ("MoE
// Architecture" s3) and the load statistics ("MoE Architecture" s2).
//
// A one-token step reads the touched experts' weights and little else (the
// handbook's Inference view), and the general path's chain of dependent
// launches -- router + grouping, up GEMM, down GEMM, combine -- costs a sixth
// of such a call in launch and dependency latency.  Here:
//  * Every CTA of both kernels routes the token itself (at most 32 dots of
//    length d; W_g comes from L2 after the first CTA), with the thread mapping
//    and addition order of the one-block-per-token router, so its ids, gates
//    and statistics are that router's bit for bit and no launch separates the
//    routing from the weight stream.
//  * Both kernels are one CTA per SM: a producer warp fills a ring of
//    shared-memory stages with 1-D bulk copies of whole weight rows (few
//    large copies: the copy engine's cost is per copy), and 16 consumer warps
//    each take a fixed slice of every row.  A lane therefore meets the same
//    activation positions in every row, and holds those activations in
//    registers: shared memory carries each weight byte once and nothing else.
//    The dots run on the CUDA cores with fp32 accumulation (at one token the
//    MMA's N side would be padding): bf16 weights through mixed-precision
//    bf16 FMAs; E4M3 codes converted exactly to f16 pairs and multiplied by
//    f16 activation pairs, 16 products summed in f16 before they join fp32.
//  * fused_up_kernel: a stage is up_rows consecutive hidden features of one
//    touched expert (their W1 rows and W3 rows, two copies); the CTA sums its
//    warps' partial dots in a fixed order and writes
//    H[entry][f] = silu(x W1^T) * (x W3^T) in bf16 (and H_shared).
//  * fused_down_kernel: a CTA owns a block of output channels r and streams
//    W2[e][r] for every touched expert e (expert by expert; up to four rows a
//    stage), the lanes holding the expert's H values at their positions; it
//    then adds the warps' slices, the row scale (FP8) and the gates in a
//    fixed order and writes y: no Y_perm and no combine launch.
//  * The down kernel reads x, W_g, the biases and its weights before its
//    grid-dependency wait and H only after it.  The up kernel triggers its
//    dependents right after its own wait, by which time whatever wrote x has
//    completed, so the down kernel's CTAs route and fill their rings while the
//    up kernel's last CTAs finish.
#include <cuda_fp8.h>
#include <float.h>

#include <type_traits>

#include "common.cuh"
#include "route_math.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {
using namespace route_math;
using tc::globaltimer;
using tc::kDrainLimitNs;
using tc::kWaitLimitNs;
using tc::mbar_arrive;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::smem_u32;
using bf16 = __nv_bfloat16;

constexpr int kFW = 16;  // consumer warps per CTA, both kernels (warp kFW is the producer)
constexpr int kFThreads = 32 * kFW;
constexpr int kFThreadsP = kFThreads + 32;
constexpr int kFMaxStages = 16;
constexpr int kDnMaxRows = 4;    // W2 rows of one down-kernel stage, at most
// dynamic shared memory of either kernel, at most (the static part -- routing,
// barriers -- stays under 5 KB of the 227 KB a CTA may hold)
constexpr size_t kFSmemBudget = 216 * 1024;
constexpr size_t kFRingCap = 200 * 1024;  // bytes in flight per SM that saturate its share of HBM

static_assert(kFusedMaxE <= 32, "one softmax lane per expert");

// The routing of the batch as every CTA holds it.
struct FusedRoute {
    int32_t ids[kFusedMaxEntries];
    float gates[kFusedMaxEntries];
    float p[kFusedMaxT][kFusedMaxE];  // softmax rows (load statistics)
    int cnt[kFusedMaxE];              // routing decisions per expert, before the capacity cut
    int col_of[kFusedMaxEntries];     // down-kernel column of each entry; -1: dropped
    int n_exp;                        // touched experts (a kept entry), ascending ids
    int exp[kFusedMaxEntries];
    int ntok[kFusedMaxEntries];                // kept entries of each, in token order
    int tok[kFusedMaxEntries][kFusedMaxT];     // their tokens
    int ent[kFusedMaxEntries][kFusedMaxT];     // their entries t k + slot (H rows)
    int col0[kFusedMaxEntries];                // first column of each expert
    int ncol;                                  // kept entries; the shared expert's T columns follow
};

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

// Routes the batch into `r` (all threads of the CTA; ends synchronised).  The
// logits are the one-block-per-token router's sums: that kernel's 512
// threads each take 16-byte vectors v = tid, tid + 512, ... of x and W_g and
// the 16 warps' butterfly sums are added in warp order; the consumer threads
// here play those 512 threads (each kSplitDThreads / kFThreads of them, with
// separate partials), so every logit is the same fp32 operations.
template <int NE>
__device__ void fused_route(const FusedDecodeArgs& a, FusedRoute& r, float (*s_red)[NE]) {
    static_assert(kFThreads % 32 == 0 && kSplitDThreads % kFThreads == 0, "whole virtual router threads");
    constexpr int V = kSplitDThreads / kFThreads;  // virtual router threads per consumer thread
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = a.d / 8;
    const uint4* w = reinterpret_cast<const uint4*>(a.wg);
    for (int t = 0; t < a.T; ++t) {
        const uint4* xr = reinterpret_cast<const uint4*>(a.x) + (size_t)t * nv;
        float acc[V][NE];
#pragma unroll
        for (int h = 0; h < V; ++h)
#pragma unroll
            for (int e = 0; e < NE; ++e) acc[h][e] = 0.f;
#pragma unroll
        for (int h = 0; h < V; ++h) {
            // the producer warp (threads kFThreads..) only meets the barriers
            const int v_end = warp < kFW ? nv : 0;
            for (int v = threadIdx.x + kFThreads * h; v < v_end; v += kSplitDThreads) {
                // bf16 pairs into mixed-precision FMAs: the router's sums, bit for bit
                const uint4 x4 = __ldcg(xr + v);
                const uint32_t xd[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    if (e < a.E) {
                        const uint4 w4 = __ldg(w + (size_t)e * nv + v);
                        const uint32_t wd[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[h][e] = fma2_bf16(xd[j], wd[j], acc[h][e]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < V; ++h)
#pragma unroll
            for (int e = 0; e < NE; ++e) {
                const float v = warp_sum(acc[h][e]);
                if (lane == 0 && warp < kFW) s_red[warp + kFW * h][e] = v;
            }
        __syncthreads();
        if (warp == 0) {
            float l[1] = {-FLT_MAX};
            if (lane < a.E) {
                float v = 0.f;
                for (int q = 0; q < kSplitDThreads / 32; ++q) v += s_red[q][lane];  // the router's fixed order
                l[0] = v + (a.logit_bias ? __ldg(a.logit_bias + lane) : 0.f);
            }
            float psum[1] = {0.f};
            int hcnt[1] = {0};
            softmax_topk<1>(t, a.E, a.k, l, a.select_bias, a.renormalize, r.ids, r.gates, psum, hcnt, nullptr);
            if (lane < a.E) r.p[t][lane] = psum[0];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        // capacity cut: an entry's rank is the number of earlier tokens that
        // chose its expert (a token's k ids are distinct)
        const int n = a.T * a.k;
        for (int e = 0; e < a.E; ++e) r.cnt[e] = 0;
        for (int j = 0; j < n; ++j) {
            const int e = r.ids[j];
            if (e < 0 || e >= a.E) {
                record_status(a.status, kStatusBounds);
                r.col_of[j] = -1;
                continue;
            }
            const int rank = r.cnt[e]++;
            r.col_of[j] = (a.capacity < 0 || rank < a.capacity) ? 0 : -1;
        }
        int ne = 0, col = 0;
        for (int e = 0; e < a.E; ++e) {
            int nt = 0;
            for (int j = 0; j < n; ++j)
                if (r.ids[j] == e && r.col_of[j] >= 0) {
                    r.tok[ne][nt] = j / a.k;
                    r.ent[ne][nt] = j;
                    r.col_of[j] = col + nt;
                    ++nt;
                }
            if (nt) {
                r.exp[ne] = e;
                r.ntok[ne] = nt;
                r.col0[ne] = col;
                col += nt;
                ++ne;
            }
        }
        r.n_exp = ne;
        r.ncol = col;
    }
    __syncthreads();
}

// Load statistics, the grouping scan's arithmetic in its order (thread 0).
__device__ void fused_stats(const FusedDecodeArgs& a, const FusedRoute& r) {
    if (threadIdx.x != 0) return;
    const bool want_fp = a.f || a.p || a.L;
    int kept_total = 0;
    float acc = 0.f;
    for (int e = 0; e < a.E; ++e) {
        const int cnt = r.cnt[e];
        const int kept = (a.capacity >= 0 && cnt > a.capacity) ? a.capacity : cnt;
        kept_total += kept;
        if (a.counts) a.counts[e] = cnt;
        if (a.kept) a.kept[e] = kept;
        if (want_fp) {
            float tot = 0.f;
            for (int t = 0; t < a.T; ++t) tot += r.p[t][e];
            const float pm = tot / (float)a.T;
            const float f = (float)cnt / ((float)a.T * (float)a.k);
            if (a.p) a.p[e] = pm;
            if (a.f) a.f[e] = f;
            acc += f * pm;
        }
    }
    if (a.n_dropped) *a.n_dropped = a.T * a.k - kept_total;
    if (a.L) *a.L = a.alpha * (float)a.E * acc;
}

// ---------------------------------------------------------------- the rings
// One CTA-wide ring of shared-memory stages per kernel.  Warp kFW (the
// producer) fills each stage with one or two 1-D bulk copies of whole weight
// rows, up to 32 KB each (64 KB for the down kernel's single copy): measured,
// the copies' cost is per copy (2-4 KB
// copies held an SM to ~7 million a second; one row of a 4096-wide bf16
// matrix per stage instead of two ran the up kernel 1.5x slower).  The kFW
// consumer warps each read their own slice of every stage and release it on
// the stage's `empty` barrier (kFW arrivals).
struct Ring {
    uint64_t full[kFMaxStages];
    uint64_t empty[kFMaxStages];
    int abort_flag;
};

__device__ __forceinline__ void ring_init(Ring& g, int S) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&g.full[s], 1);
            mbar_init(&g.empty[s], kFW);
        }
        g.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
}

// After a wait gave up (the producer thread): wait, bounded, for the copies of
// the last min(S, issued) items -- the only ones that may still be landing.
__device__ __forceinline__ void ring_drain(Ring& g, int S, int issued) {
    volatile int no_abort = 0;
    for (int j = issued > S ? issued - S : 0; j < issued; ++j)
        mbar_wait(&g.full[j % S], (uint32_t)((j / S) & 1), &no_abort, nullptr, kDrainLimitNs);
}

// ---------------------------------------------------------------- up kernel

// Activations live in registers: a consumer lane always reads the same
// PV vectors of every weight row it streams (16-byte vectors lane + 32 i
// of its warp's slice), so the x (or H) values those meet are loaded once
// per token (per expert, in the down kernel) and shared memory carries
// only the weights -- one read of each byte.  Against bf16 weights they stay
// bf16 pairs, multiplied by mixed-precision FMAs; against E4M3 codes they
// become f16 pairs scaled by a power of two per warp slice (the slice's
// largest magnitude lands in [0.5, 1)), multiplied with the codes as f16
// pairs.  A lane holds PV (2 or 4) vectors per token, at most kLaneWords
// registers.
constexpr int kLaneWords = 64;

// Two E4M3 codes (the low 16 bits) -> an f16 pair, exactly (E4M3 values are f16 values).
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint32_t two) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xffffu), __NV_E4M3);
    return *reinterpret_cast<const __half2*>(&hr);
}

// Activation registers per 16-byte weight vector: 4 bf16 pairs against bf16
// weights, 8 f16 pairs against E4M3 codes.
template <bool W8>
using act_t = uint32_t;
template <bool W8>
constexpr int act_n() {
    return W8 ? 8 : 4;
}

// Sums V values (1, 2 or 4) over the warp's 32 lanes at once: each butterfly
// step first exchanges halves of the value set, so V sums take 5, 5 and 6
// shuffles instead of 5 V.  Value i ends in lanes [i 32/V, (i+1) 32/V); each
// lane returns the sum of its value.  Fixed order: deterministic.
template <int V>
__device__ __forceinline__ float warp_sum_multi(const float (&x)[V]) {

    static_assert(V == 1 || V == 2 || V == 4, "1, 2 or 4 values");
    const int lane = threadIdx.x & 31;
    float v;
    if constexpr (V == 1) {
        v = x[0] + __shfl_xor_sync(0xffffffffu, x[0], 16);
    } else if constexpr (V == 2) {
        const bool b4 = lane & 16;
        v = (b4 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, b4 ? x[0] : x[1], 16);
    } else {
        const bool b4 = lane & 16, b3 = lane & 8;
        const float p0 = (b4 ? x[2] : x[0]) + __shfl_xor_sync(0xffffffffu, b4 ? x[0] : x[2], 16);
        const float p1 = (b4 ? x[3] : x[1]) + __shfl_xor_sync(0xffffffffu, b4 ? x[1] : x[3], 16);
        v = (b3 ? p1 : p0) + __shfl_xor_sync(0xffffffffu, b3 ? p0 : p1, 8);
    }
#pragma unroll
    for (int o = V == 4 ? 4 : 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The lane's activations of one token row at its PV vectors (v = lane + 32 i,
// i < PV) of the slice [a0, a0 + n), zero past the slice; bf16 pairs as they
// are against bf16 weights.  FP8: returned as f16 pairs of x 2^-e, e chosen for the whole
// warp so that the slice's largest magnitude lands in [0.5, 1) (e = 0 for an
// all-zero slice; e kept in [-125, 126]); the return value is 2^e, which the warp's dots are
// multiplied by (exactly: a power of two).  Must be called by whole warps.
template <bool W8, int PV>
__device__ __forceinline__ float load_act(const bf16* row, int a0, int n, act_t<W8> (&out)[PV][act_n<W8>()]) {
    constexpr int VE = W8 ? 16 : 8;
    const int lane = threadIdx.x & 31;
    if constexpr (W8) {
        float xv[PV][16];
        uint32_t mx = 0;  // largest |x| of the lane, as bits (same order as the values)
#pragma unroll
        for (int i = 0; i < PV; ++i) {
            const int v = lane + 32 * i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint4 u = make_uint4(0u, 0u, 0u, 0u);
                if (v * VE < n) u = __ldcg(reinterpret_cast<const uint4*>(row + a0 + v * VE) + h);
                float f8[8];
                widen(u, f8, static_cast<const __nv_bfloat16*>(nullptr));
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    xv[i][8 * h + e] = f8[e];
                    mx = max(mx, __float_as_uint(fabsf(f8[e])));
                }
            }
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        int ex = 0;
        if (mx != 0) frexpf(__uint_as_float(mx), &ex);  // max = m 2^ex, m in [0.5, 1)
        // both 2^-ex and 2^ex stay finite fp32 values: at the ends of the bf16
        // range the slice's largest magnitude then lands below 4 (f16 sums of
        // eight products stay below 8 x 448 x 4) or below 0.5
        ex = ex < -125 ? -125 : (ex > 126 ? 126 : ex);
        const float scale = ldexpf(1.0f, -ex);
#pragma unroll
        for (int i = 0; i < PV; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const __half2 p2 = __floats2half2_rn(xv[i][2 * e] * scale, xv[i][2 * e + 1] * scale);
                out[i][e] = *reinterpret_cast<const uint32_t*>(&p2);
            }
        return ldexpf(1.0f, ex);
    } else {
#pragma unroll
        for (int i = 0; i < PV; ++i) {
            const int v = lane + 32 * i;
            uint4 u = make_uint4(0u, 0u, 0u, 0u);
            if (v * VE < n) u = __ldcg(reinterpret_cast<const uint4*>(row + a0 + v * VE));
            out[i][0] = u.x;
            out[i][1] = u.y;
            out[i][2] = u.z;
            out[i][3] = u.w;
        }
        return 1.0f;
    }
}

// acc[q][i] += <activations of token q, 16-byte weight vector lane + 32 i of
// the slice at `w`> for the vectors below nvec.  E4M3 codes: the 16 products
// of a vector are summed as f16 pairs (two partial sums of 8 products each,
// |sum| < 8 x 448 with activations below 1), which then join the fp32
// accumulator.
template <bool W8, int NT, int PV>
__device__ __forceinline__ void slice_dots(const uint8_t* w, int nvec, const act_t<W8> (&act)[NT][PV][act_n<W8>()],
                                           int ntok, float (&acc)[NT][PV]) {
    const int lane = threadIdx.x & 31;
    const uint4* wv = reinterpret_cast<const uint4*>(w);
#pragma unroll
    for (int i = 0; i < PV; ++i) {
        const int v = lane + 32 * i;
        if (v < nvec) {
            const uint4 u = wv[v];
            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
            if constexpr (W8) {
                __half2 wh[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    wh[2 * j] = e4m3x2_to_half2(wd[j]);
                    wh[2 * j + 1] = e4m3x2_to_half2(wd[j] >> 16);
                }
#pragma unroll
                for (int q = 0; q < NT; ++q)
                    if (q < ntok) {
                        __half2 s2 = __float2half2_rn(0.0f);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            s2 = __hfma2(wh[e], *reinterpret_cast<const __half2*>(&act[q][i][e]), s2);
                        const float2 f = __half22float2(s2);
                        acc[q][i] += f.x + f.y;
                    }
            } else {
#pragma unroll
                for (int q = 0; q < NT; ++q)
                    if (q < ntok) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[q][i] = fma2_bf16(wd[j], act[q][i][j], acc[q][i]);
                    }
            }
        }
    }
}

// The up kernel's work list: blocks of up_rows consecutive hidden features
// of one touched expert (expert slot es < n_exp) or of the shared expert (es
// == n_exp), expert-major; block b goes to CTA b mod grid.  A stage holds one
// block's whole rows of W1 and of W3 (two bulk copies); consumer warp w works
// on row w / (kFW / up_rows) of the block, on slice w mod (kFW / up_rows) of d.
struct UpCursor {
    int es, f;  // expert slot, first feature of the block
};

template <bool W8, int NT, int NE, int PV>
__global__ void __launch_bounds__(kFThreadsP, 1)
    fused_up_kernel(const FusedDecodeArgs a, const FusedPlan pl, int stall, uint64_t wait_ns) {
    constexpr int WB = W8 ? 1 : 2;
    constexpr int VE = W8 ? 16 : 8;  // elements per 16-byte weight vector
    static_assert(NT * PV * act_n<W8>() <= kLaneWords, "activation registers");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ FusedRoute r;
    __shared__ float s_red[kSplitDThreads / 32][NE];
    __shared__ __align__(8) Ring g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = pl.up_stages;
    ring_init(g, S);
    __syncthreads();
    pdl_wait();
    // the down kernel reads nothing of this kernel's before its own wait
    pdl_trigger();
    fused_route<NE>(a, r, s_red);
    if (blockIdx.x == 0) fused_stats(a, r);
    const int d = a.d, F = a.F, Fs = a.Fs, n_exp = r.n_exp;
    float* part = reinterpret_cast<float*>(smem);  // [block][row][warp of row][T][2]: x.W1, x.W3
    uint8_t* ring = smem + pl.up_part_bytes;
    const int R = pl.up_rows;
    const int nb = (F + R - 1) / R, nbs = a.n_shared ? (Fs + R - 1) / R : 0;
    const int n_all = n_exp * nb + nbs;
    const int grid = gridDim.x;
    const int n_blocks = (int)blockIdx.x < n_all ? (n_all - (int)blockIdx.x + grid - 1) / grid : 0;
    const size_t mat_bytes = (size_t)R * d * WB;  // one matrix's rows in a stage
    auto start = [&](UpCursor& k) {
        const int b = blockIdx.x;
        k.es = b / nb < n_exp ? b / nb : n_exp;
        k.f = (b - k.es * nb) * R;
    };
    auto advance = [&](UpCursor& k) {
        int fb = k.f / R + grid;
        while (k.es < n_exp && fb >= nb) {
            fb -= nb;
            ++k.es;
        }
        k.f = fb * R;
    };
    int issued = 0;
    if (warp == kFW) {
        // ---- producer ----
        if (lane == 0 && !stall) {
            UpCursor k;
            start(k);
            int s = 0;
            uint32_t ph = 0;
            for (; issued < n_blocks; ++issued) {
                if (!mbar_wait(&g.empty[s], ph ^ 1u, &g.abort_flag, a.status, wait_ns)) break;
                const bool routed = k.es < n_exp;
                const int Fe = routed ? F : Fs;
                const size_t row0 = routed ? (size_t)r.exp[k.es] * F + k.f : (size_t)k.f;
                const int rv = Fe - k.f < R ? Fe - k.f : R;
                const uint32_t bytes = (uint32_t)((size_t)rv * d * WB);
                uint8_t* dst = ring + (size_t)s * 2 * mat_bytes;
                mbar_expect_tx(&g.full[s], 2 * bytes);
                bulk_g2s(dst, static_cast<const uint8_t*>(routed ? a.w1 : a.ws1) + row0 * d * WB, bytes,
                         &g.full[s]);
                bulk_g2s(dst + mat_bytes, static_cast<const uint8_t*>(routed ? a.w3 : a.ws3) + row0 * d * WB, bytes,
                         &g.full[s]);
                advance(k);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else {
        // ---- consumers: row j of each block, slice `sub` of d ----
        const int wpr = kFW / R, j = warp / wpr, sub = warp % wpr;
        const int a0 = sub * pl.up_wslice;
        const int n = d - a0 < pl.up_wslice ? (d - a0 > 0 ? d - a0 : 0) : pl.up_wslice;
        const int nvec = n / VE;
        act_t<W8> xr[NT][PV][act_n<W8>()];  // every token's x at this lane's positions
        float xs[NT];                        // ... and the factor its dots take (FP8: 2^e)
#pragma unroll
        for (int q = 0; q < NT; ++q) {
            xs[q] = 1.0f;
            if (q < a.T) {
                xs[q] = load_act<W8, PV>(static_cast<const bf16*>(a.x) + (size_t)q * d, a0, n, xr[q]);
            } else {
#pragma unroll
                for (int i = 0; i < PV; ++i)
#pragma unroll
                    for (int e = 0; e < act_n<W8>(); ++e) xr[q][i][e] = 0;
            }
        }
        // Every block's dots are taken with all T tokens (at most kFusedMaxT);
        // the reduction below keeps those of the tokens that chose the expert.
        UpCursor k;
        start(k);
        int s = 0;
        uint32_t ph = 0;
        for (int bl = 0; bl < n_blocks; ++bl) {
            const bool routed = k.es < n_exp;
            if (!mbar_wait(&g.full[s], ph, &g.abort_flag, a.status, wait_ns)) break;
            const bool row_ok = k.f + j < (routed ? F : Fs);
            float gacc[NT][PV], uacc[NT][PV];
#pragma unroll
            for (int q = 0; q < NT; ++q)
#pragma unroll
                for (int i = 0; i < PV; ++i) gacc[q][i] = uacc[q][i] = 0.f;
            if (row_ok && nvec > 0) {
                const uint8_t* w1 = ring + (size_t)s * 2 * mat_bytes + ((size_t)j * d + a0) * WB;
                slice_dots<W8, NT, PV>(w1, nvec, xr, a.T, gacc);
                slice_dots<W8, NT, PV>(w1 + mat_bytes, nvec, xr, a.T, uacc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&g.empty[s]);
            if (row_ok) {
                float vals[2 * NT];  // x.W1 and x.W3 of each token
#pragma unroll
                for (int q = 0; q < NT; ++q) {
                    vals[2 * q] = vals[2 * q + 1] = 0.f;
#pragma unroll
                    for (int i = 0; i < PV; ++i) {
                        vals[2 * q] += gacc[q][i];
                        vals[2 * q + 1] += uacc[q][i];
                    }
                }
                float tot = warp_sum_multi<2 * NT>(vals);
                constexpr int kPer = 32 / (2 * NT);  // lanes per value
                const int vi = lane / kPer;
#pragma unroll
                for (int q = 0; q < NT; ++q)
                    if (q == (vi >> 1)) tot *= xs[q];
                if (lane % kPer == 0 && (vi >> 1) < a.T)
                    part[((((size_t)bl * R + j) * wpr + sub) * a.T + (vi >> 1)) * 2 + (vi & 1)] = tot;
            }
            advance(k);
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
    }
    __syncthreads();
    if (g.abort_flag) {
        if (warp == kFW && lane == 0 && !stall) ring_drain(g, S, issued);
        return;
    }
    // H = silu(x W1^T) * (x W3^T): each (block, row, token of the expert)
    // adds its row's warps' partials in warp order
    const int wpr = kFW / R;
    for (int idx = threadIdx.x; idx < n_blocks * R * a.T; idx += blockDim.x) {
        const int i = idx % a.T, jr = (idx / a.T) % R, bl = idx / (a.T * R);
        const int b = (int)blockIdx.x + bl * grid;
        const bool routed = b < n_exp * nb;
        const int es = routed ? b / nb : n_exp;
        const int f = (routed ? b - es * nb : b - n_exp * nb) * R + jr;
        if (f >= (routed ? F : Fs) || i >= (routed ? r.ntok[es] : a.T)) continue;
        const int t = routed ? r.tok[es][i] : i;
        float gv = 0.f, uv = 0.f;
        for (int sub = 0; sub < wpr; ++sub) {
            const float* p = part + ((((size_t)bl * R + jr) * wpr + sub) * a.T + t) * 2;
            gv += p[0];
            uv += p[1];
        }
        if (W8) {
            gv *= routed ? __ldg(a.s1 + (size_t)r.exp[es] * F + f) : __ldg(a.ss1 + f);
            uv *= routed ? __ldg(a.s3 + (size_t)r.exp[es] * F + f) : __ldg(a.ss3 + f);
        }
        const bf16 h = __float2bfloat16_rn(silu_mul(gv, uv));
        if (routed)
            static_cast<bf16*>(a.h)[(size_t)r.ent[es][i] * F + f] = h;
        else
            static_cast<bf16*>(a.h_shared)[(size_t)i * Fs + f] = h;
    }
}

// ---------------------------------------------------------------- down kernel

// The down kernel's work list for one CTA's output channels r0..r1: expert
// slot es (n_exp: the shared expert), then channels, dn_rows_stage (1 to
// kDnMaxRows) whole consecutive W2 rows per stage (one bulk copy).  Consumer warp w takes
// slice [w cs, w cs + cs) of every row, its lanes the same positions in each,
// so the expert's tokens' H values there are loaded into registers once per
// expert.
template <bool W8, int NT, int NE, int PV>
__global__ void __launch_bounds__(kFThreadsP, 1)
    fused_down_kernel(const FusedDecodeArgs a, const FusedPlan pl, int stall, uint64_t wait_ns) {
    constexpr int WB = W8 ? 1 : 2;
    constexpr int VE = W8 ? 16 : 8;
    static_assert(NT * PV * act_n<W8>() <= kLaneWords, "activation registers");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ FusedRoute r;
    __shared__ float s_red[kSplitDThreads / 32][NE];
    __shared__ __align__(8) Ring g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = pl.dn_stages;
    ring_init(g, S);
    __syncthreads();
    // Before the grid-dependency wait: x, W_g, the biases and W2 only.  This
    // launch starts after every CTA of the up kernel passed its own wait, so
    // whatever wrote x has completed; x is read through L2.
    fused_route<NE>(a, r, s_red);

    const int d = a.d, F = a.F, Fs = a.Fs, n_exp = r.n_exp;
    const int r0 = (int)((long long)blockIdx.x * d / gridDim.x);
    const int r1 = (int)((long long)(blockIdx.x + 1) * d / gridDim.x);
    const int nr = r1 - r0;
    const int R2 = pl.dn_rows_stage;
    const int per_exp = (nr + R2 - 1) / R2;  // stages per expert
    const int n_items = (n_exp + (a.n_shared ? 1 : 0)) * per_exp;
    const int ncols = r.ncol + (a.n_shared ? a.T : 0);
    float* part = reinterpret_cast<float*>(smem);  // [kFW][nr][ncols]
    uint8_t* ring = smem + pl.dn_part_bytes;
    const size_t stage_bytes = pl.dn_stage_bytes;
    int issued = 0;
    if (warp == kFW) {
        // ---- producer: weights only, so it starts before the up kernel has finished ----
        if (lane == 0 && !stall) {
            int es = 0, row = 0, s = 0;
            uint32_t ph = 0;
            for (; issued < n_items; ++issued) {
                if (!mbar_wait(&g.empty[s], ph ^ 1u, &g.abort_flag, a.status, wait_ns)) break;
                const bool routed = es < n_exp;
                const uint8_t* src =
                    routed ? static_cast<const uint8_t*>(a.w2) + ((size_t)r.exp[es] * d + (r0 + row)) * F * WB
                           : static_cast<const uint8_t*>(a.ws2) + (size_t)(r0 + row) * Fs * WB;
                const int rows = nr - row < R2 ? nr - row : R2;
                const uint32_t bytes = (uint32_t)(rows * (routed ? F : Fs) * WB);
                mbar_expect_tx(&g.full[s], bytes);
                bulk_g2s(ring + (size_t)s * stage_bytes, src, bytes, &g.full[s]);
                row += R2;
                if (row >= nr) {
                    row = 0;
                    ++es;
                }
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else {
        // ---- consumers ----
        for (int i = lane; i < nr * ncols; i += 32) part[(size_t)warp * nr * ncols + i] = 0.f;
        pdl_wait();  // H from here on
        act_t<W8> h[NT][PV][act_n<W8>()];  // the current expert's tokens' H at this lane's positions
        float hs[NT];                       // ... and the factor their dots take (FP8: 2^e)
        int es = 0, row = 0, s = 0, cur_es = -1, ntok = 0, col0 = 0, a0 = 0, nvec = 0, Fe = 0;
        uint32_t ph = 0;
        for (int q = 0; q < n_items; ++q) {
            const bool routed = es < n_exp;
            if (es != cur_es) {
                cur_es = es;
                ntok = routed ? r.ntok[es] : a.T;
                col0 = routed ? r.col0[es] : r.ncol;
                const int cs = routed ? pl.dn_wslice : pl.dn_wslice_s;
                Fe = routed ? F : Fs;
                a0 = warp * cs;
                const int n = Fe - a0 < cs ? (Fe - a0 > 0 ? Fe - a0 : 0) : cs;
                nvec = n / VE;
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    hs[i] = 1.0f;
                    if (i < ntok) {
                        const bf16* hrow = routed ? static_cast<const bf16*>(a.h) + (size_t)r.ent[es][i] * F
                                                  : static_cast<const bf16*>(a.h_shared) + (size_t)i * Fs;
                        hs[i] = load_act<W8, PV>(hrow, a0, n, h[i]);
                    }
                }
            }
            if (!mbar_wait(&g.full[s], ph, &g.abort_flag, a.status, wait_ns)) break;
            const int rows = nr - row < R2 ? nr - row : R2;
            float acc[kDnMaxRows][NT][PV];  // [row of the stage][token][vector]
#pragma unroll
            for (int jj = 0; jj < kDnMaxRows; ++jj)
#pragma unroll
                for (int i = 0; i < NT; ++i)
#pragma unroll
                    for (int v = 0; v < PV; ++v) acc[jj][i][v] = 0.f;
            if (nvec > 0) {
                const uint8_t* st = ring + (size_t)s * stage_bytes + (size_t)a0 * WB;
#pragma unroll
                for (int jj = 0; jj < kDnMaxRows; ++jj)
                    if (jj < rows) slice_dots<W8, NT, PV>(st + (size_t)jj * Fe * WB, nvec, h, ntok, acc[jj]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&g.empty[s]);
            float vals[kDnMaxRows * NT];  // (row, token) dots
#pragma unroll
            for (int jj = 0; jj < kDnMaxRows; ++jj)
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    vals[jj * NT + i] = 0.f;
#pragma unroll
                    for (int v = 0; v < PV; ++v) vals[jj * NT + i] += acc[jj][i][v];
                }
            float tot = warp_sum_multi<kDnMaxRows * NT>(vals);
            constexpr int kPer = 32 / (kDnMaxRows * NT);  // lanes per value
            const int vi = lane / kPer, jj = vi / NT, ti = vi % NT;
#pragma unroll
            for (int i = 0; i < NT; ++i)
                if (i == ti) tot *= hs[i];
            if (lane % kPer == 0 && jj < rows && ti < ntok) part[((size_t)warp * nr + row + jj) * ncols + col0 + ti] = tot;
            row += R2;
            if (row >= nr) {
                row = 0;
                ++es;
            }
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
    }
    __syncthreads();
    if (g.abort_flag) {
        if (warp == kFW && lane == 0 && !stall) ring_drain(g, S, issued);
        return;
    }

    // y[t][r] = sum over the token's kept slots (slot order) of g_j * (scale * slices)
    //           + the shared expert's slices
    for (int idx = threadIdx.x; idx < nr * a.T; idx += blockDim.x) {
        const int row = idx / a.T, t = idx % a.T;
        const int rr = r0 + row;
        float y = 0.f;
        for (int sl = 0; sl < a.k; ++sl) {
            const int j = t * a.k + sl;
            const int col = r.col_of[j];
            if (col < 0) continue;
            float v = 0.f;
            for (int w = 0; w < kFW; ++w) v += part[((size_t)w * nr + row) * ncols + col];
            if (W8) v *= __ldg(a.s2 + (size_t)r.ids[j] * d + rr);
            y += r.gates[j] * v;
        }
        if (a.n_shared) {
            float v = 0.f;
            for (int w = 0; w < kFW; ++w) v += part[((size_t)w * nr + row) * ncols + r.ncol + t];
            if (W8) v *= __ldg(a.ss2 + rr);
            y += v;
        }
        if (a.y_fp32)
            static_cast<float*>(a.y)[(size_t)t * d + rr] = y;
        else
            static_cast<bf16*>(a.y)[(size_t)t * d + rr] = __float2bfloat16_rn(y);
    }
}

size_t align128(size_t v) { return (v + 127) / 128 * 128; }

template <typename K>
cudaError_t set_smem_once(K kernel, uint64_t& mask) {
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit && (mask & bit)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFSmemBudget);
    if (e == cudaSuccess) mask |= bit;
    return e;
}

template <bool UP, bool W8, int NT, int NE, int PV>
cudaError_t launch_one(const FusedDecodeArgs& a, const FusedPlan& p, cudaStream_t s) {
    static uint64_t mask = 0;
    const int stall = test_stall_gemm() ? 1 : 0;
    const uint64_t wait_ns = stall ? kStallWaitLimitNs : kWaitLimitNs;
    if constexpr (NT * PV * act_n<W8>() > kLaneWords) {
        return cudaErrorInvalidValue;  // never planned
    } else if constexpr (UP) {
        const cudaError_t e = set_smem_once(fused_up_kernel<W8, NT, NE, PV>, mask);
        if (e != cudaSuccess) return e;
        return launch_pdl(fused_up_kernel<W8, NT, NE, PV>, dim3(p.grid_up), dim3(kFThreadsP), p.up_smem, s, a, p,
                          stall, wait_ns);
    } else {
        const cudaError_t e = set_smem_once(fused_down_kernel<W8, NT, NE, PV>, mask);
        if (e != cudaSuccess) return e;
        return launch_pdl(fused_down_kernel<W8, NT, NE, PV>, dim3(p.grid_dn), dim3(kFThreadsP), p.dn_smem, s, a, p,
                          stall, wait_ns);
    }
}

template <bool UP, bool W8, int NT, int NE>
cudaError_t launch_pv(const FusedDecodeArgs& a, const FusedPlan& p, cudaStream_t s) {
    return (UP ? p.up_pv : p.dn_pv) == 2 ? launch_one<UP, W8, NT, NE, 2>(a, p, s) : launch_one<UP, W8, NT, NE, 4>(a, p, s);
}

template <bool UP, bool W8>
cudaError_t launch_nt(const FusedDecodeArgs& a, const FusedPlan& p, cudaStream_t s) {
    static_assert(kFusedMaxT == 1, "instantiated for one token");
    return a.E <= 8 ? launch_pv<UP, W8, 1, 8>(a, p, s) : launch_pv<UP, W8, 1, 32>(a, p, s);
}

}  // namespace

FusedPlan fused_decode_plan(const moe_config& c, bool fp8, int sms) {
    FusedPlan p{};
    p.ok = false;
    if (c.routing != MOE_ROUTE_TOKEN_CHOICE || c.dtype != MOE_BF16 || c.h_split != 0) return p;
    if (c.T < 1 || c.T > kFusedMaxT || c.E > kFusedMaxE || (long long)c.T * c.k > kFusedMaxEntries) return p;
    if (sms < 1) return p;
    const int wb = fp8 ? 1 : 2, ve = fp8 ? 16 : 8;  // bytes per weight; elements per 16-byte vector
    const int T = c.T;
    // bytes of one bulk copy (one stage), at most, unless one row is longer
    const int kCopyUp = 32768, kCopyDn = 65536;
    // activation vectors per lane for a warp slice: 2 or 4, within kLaneWords registers
    auto pv_of = [&](int slice) {
        const int v = (slice + 32 * ve - 1) / (32 * ve);
        const int pv = v <= 2 ? 2 : 4;
        return v <= 4 && T * pv * (fp8 ? 8 : 4) <= kLaneWords ? pv : 0;
    };
    auto round_up = [](int v, int m) { return (v + m - 1) / m * m; };
    // up kernel: the partial dots, then the ring; a stage holds up_rows whole
    // rows of W1 and of W3
    auto wslice = [&](int rows) { return round_up((c.d + kFW / rows - 1) / (kFW / rows), ve); };
    p.up_rows = 1;
    while (p.up_rows * 2 <= kFW && (long long)p.up_rows * 2 * c.d * wb <= kCopyUp && pv_of(wslice(p.up_rows * 2)))
        p.up_rows *= 2;
    p.up_wslice = wslice(p.up_rows);
    p.up_pv = pv_of(p.up_wslice);
    if (!p.up_pv) return p;
    p.grid_up = sms;
    const long long touched = (long long)T * c.k < c.E ? (long long)T * c.k : c.E;
    const long long blocks = touched * ((c.d_ff + p.up_rows - 1) / p.up_rows) +
                             (c.n_shared ? (c.d_ff_shared + p.up_rows - 1) / p.up_rows : 0);
    const long long blocks_cta = (blocks + sms - 1) / sms;
    p.up_part_bytes = align128((size_t)blocks_cta * kFW * T * 8);
    const size_t up_stage = (size_t)2 * p.up_rows * c.d * wb;
    if (p.up_part_bytes + 2 * up_stage > kFSmemBudget) return p;
    size_t ring = kFSmemBudget - p.up_part_bytes;
    if (ring > kFRingCap) ring = kFRingCap;
    p.up_stages = (int)(ring / up_stage);
    if (p.up_stages < 2) p.up_stages = 2;
    if (p.up_stages > kFMaxStages) p.up_stages = kFMaxStages;
    p.up_smem = p.up_part_bytes + (size_t)p.up_stages * up_stage;
    // down kernel: the partial dots, then the ring of whole W2 rows
    p.dn_wslice = round_up((c.d_ff + kFW - 1) / kFW, ve);
    p.dn_wslice_s = c.n_shared ? round_up((c.d_ff_shared + kFW - 1) / kFW, ve) : 0;
    p.dn_pv = pv_of(p.dn_wslice > p.dn_wslice_s ? p.dn_wslice : p.dn_wslice_s);
    if (!p.dn_pv) return p;
    const int fmax = c.n_shared && c.d_ff_shared > c.d_ff ? c.d_ff_shared : c.d_ff;
    p.dn_rows_stage = 1;
    while (p.dn_rows_stage * 2 <= kDnMaxRows && (long long)p.dn_rows_stage * 2 * fmax * wb <= kCopyDn)
        p.dn_rows_stage *= 2;
    p.dn_stage_bytes = align128((size_t)p.dn_rows_stage * fmax * wb);
    p.grid_dn = sms < c.d ? sms : c.d;
    p.dn_rows = (c.d + p.grid_dn - 1) / p.grid_dn;
    p.dn_cols = T * c.k + (c.n_shared ? T : 0);
    p.dn_part_bytes = align128((size_t)kFW * p.dn_rows * p.dn_cols * 4);
    if (p.dn_part_bytes + 2 * p.dn_stage_bytes > kFSmemBudget) return p;
    ring = kFSmemBudget - p.dn_part_bytes;
    if (ring > kFRingCap) ring = kFRingCap;
    p.dn_stages = (int)(ring / p.dn_stage_bytes);
    if (p.dn_stages < 2) p.dn_stages = 2;
    if (p.dn_stages > kFMaxStages) p.dn_stages = kFMaxStages;
    p.dn_smem = p.dn_part_bytes + (size_t)p.dn_stages * p.dn_stage_bytes;
    p.ok = true;
    return p;
}

cudaError_t launch_fused_up(const FusedDecodeArgs& a, const FusedPlan& p, cudaStream_t s) {
    if (!p.ok || a.T < 1 || a.T > kFusedMaxT || a.E > kFusedMaxE) return cudaErrorInvalidValue;
    return a.fp8 ? launch_nt<true, true>(a, p, s) : launch_nt<true, false>(a, p, s);
}

cudaError_t launch_fused_down(const FusedDecodeArgs& a, const FusedPlan& p, cudaStream_t s) {
    if (!p.ok || a.T < 1 || a.T > kFusedMaxT || a.E > kFusedMaxE) return cudaErrorInvalidValue;
    return a.fp8 ? launch_nt<false, true>(a, p, s) : launch_nt<false, false>(a, p, s);
}

}  // namespace moe
