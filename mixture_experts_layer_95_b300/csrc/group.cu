// group.cu -- grouping of the (token, slot) entries by expert.
//
// "Mixture of experts (MoE)" handbook, "Implementation: token by token vs.
// grouped by expert": flatten the entries in order t*k + j, sort them by
// expert with a stable sort, count each expert (bincount) and give each a
// running start (a prefix sum).  Capacity ("Mixture of Experts" notes, How it
// works; "MoE Architecture" s2): an expert keeps its first C entries in that
// order and drops the rest.
//
// GPU form (reduce-then-scan, no spin-waits):
//  1. a shared-memory histogram of the chosen ids per chunk of tokens
//     (emitted by the router for free, or by group_hist_kernel) ->
//     block_hist [nchunk][E];
//  2. group_scan_kernel: every block re-reads the whole (small) block_hist,
//     derives the global counts, the capacity cut, the expert offsets and its
//     own per-expert starting ranks, then ranks its entries stably with warp
//     match/popc and writes slot_pos, sorted_token_ids and gates_perm.
//     Every expert's base offset depends on all tokens, so a decoupled
//     look-back would not save the second pass; the redundant per-block scan
//     of a few KB keeps the kernel free of inter-block waits.
//  3. gather_rows_kernel copies x rows into expert order with 16-byte vectors.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;
// The load statistics keep the order moe_load_stats uses (warp columns only
// up to kWarpColumnMaxE).

__global__ void __launch_bounds__(kRouterThreads) group_hist_kernel(int Tn, int E, int k, int chunk,
                                                                     const int32_t* __restrict__ ids,
                                                                     int32_t* __restrict__ block_hist,
                                                                     int* status) {
    pdl_wait();
    extern __shared__ int s_hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();
    const size_t n = (size_t)Tn * k;
    const size_t lo = (size_t)blockIdx.x * chunk * k;
    const size_t hi = min(n, lo + (size_t)chunk * k);
    for (size_t i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        const int e = ids[i];
        if (e < 0 || e >= E) {
            record_status(status, kStatusBounds);
            continue;
        }
        atomicAdd(&s_hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) block_hist[(size_t)blockIdx.x * E + e] = s_hist[e];
    __syncthreads();
    pdl_trigger();
}

// Exclusive scan over v[0..n) in shared memory (n <= kMaxExperts), result in
// out[0..n] with out[n] = total.  Called by all threads of the block.
__device__ void block_exclusive_scan(const int* v, int* out, int n, int* s_warp) {
    const int per = (n + kScanThreads - 1) / kScanThreads;  // <= 4
    const int b = threadIdx.x * per;
    int local = 0;
    for (int i = 0; i < per; ++i)
        if (b + i < n) local += v[b + i];
    // warp-level inclusive scan of the per-thread sums
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int w = 0; w < kScanWarps; ++w) {
            const int t = s_warp[w];
            s_warp[w] = run;
            run += t;
        }
        s_warp[kScanWarps] = run;
    }
    __syncthreads();
    int run = s_warp[warp] + incl - local;
    for (int i = 0; i < per; ++i)
        if (b + i < n) {
            out[b + i] = run;
            run += v[b + i];
        }
    if (threadIdx.x == 0) out[n] = s_warp[kScanWarps];
    __syncthreads();
}

// The statistics block stages the p rows in shared memory (one coalesced
// pass) when they fit this many floats, then adds each column in row order.
constexpr int kScanStageFloats = 16384;

struct ScanArgs {
    int T, E, k, chunk, capacity, nblk;
    int p_stage;  // 1: stage o.p_part ([o.p_nblk][E]) in shared memory for the statistics
    const int32_t* ids;
    const float* gates;
    const int32_t* block_hist;
    GroupOut o;
    int* status;
};

__global__ void __launch_bounds__(kScanThreads) group_scan_kernel(const ScanArgs a) {
    pdl_wait();
    extern __shared__ int s_mem[];
    const int E = a.E;
    int* s_before = s_mem;                 // [E]   this block's starting rank per expert
    int* s_kept = s_before + E;            // [E]
    int* s_off = s_kept + E;               // [E+1]
    int* s_wcnt = s_off + E + 1;           // [kScanWarps][E]
    int* s_warp = s_wcnt + kScanWarps * E; // [kScanWarps + 1]
    float* s_red = reinterpret_cast<float*>(s_warp + kScanWarps + 1);  // [kScanThreads]
    int* s_pb = reinterpret_cast<int*>(s_red + kScanThreads);           // [kScanWarps][E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = a.T * a.k;

    // 1. global counts, this block's prefix, capacity cut.  Up to kScanThreads
    // experts: thread t = e + E j (j < cpt) sums column e over rows j, j + cpt,
    // ..., so consecutive threads read consecutive columns of a row and every
    // thread keeps 32 rows in flight; the cpt partial sums per column are then
    // added through shared memory (integers: any order gives the same counts).
    // More experts: one thread per expert walking all rows.
    if (E <= kScanThreads) {
        const int cpt = kScanThreads / E < kScanWarps ? kScanThreads / E : kScanWarps;
        if ((int)threadIdx.x < cpt * E) {
            const int e = threadIdx.x % E, j = threadIdx.x / E;
            int tot = 0, before = 0;
            for (int b0 = j; b0 < a.nblk; b0 += 32 * cpt) {
                int v[32];
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int b = b0 + u * cpt;
                    v[u] = b < a.nblk ? __ldg(a.block_hist + (size_t)b * E + e) : 0;
                }
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    tot += v[u];
                    before += (b0 + u * cpt < (int)blockIdx.x) ? v[u] : 0;
                }
            }
            s_wcnt[j * E + e] = tot;
            s_pb[j * E + e] = before;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += kScanThreads) {
            int tot = 0, before = 0;
            for (int j = 0; j < cpt; ++j) {
                tot += s_wcnt[j * E + e];
                before += s_pb[j * E + e];
            }
            s_before[e] = before;
            s_kept[e] = (a.capacity >= 0 && tot > a.capacity) ? a.capacity : tot;
            if (blockIdx.x == 0) {
                a.o.counts[e] = tot;
                a.o.kept[e] = s_kept[e];
            }
            s_wcnt[e] = tot;  // scratch: counts for the statistics below (only this thread's column)
        }
    } else {
        for (int e = threadIdx.x; e < E; e += kScanThreads) {
            int tot = 0, before = 0;
            for (int b0 = 0; b0 < a.nblk; b0 += 32) {  // 32 independent loads in flight per batch
                int v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[j] = b0 + j < a.nblk ? __ldg(a.block_hist + (size_t)(b0 + j) * E + e) : 0;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    before += (b0 + j < (int)blockIdx.x) ? v[j] : 0;
                    tot += v[j];
                }
            }
            s_before[e] = before;
            s_kept[e] = (a.capacity >= 0 && tot > a.capacity) ? a.capacity : tot;
            if (blockIdx.x == 0) {
                a.o.counts[e] = tot;
                a.o.kept[e] = s_kept[e];
            }
            s_wcnt[e] = tot;  // scratch: counts for the statistics below
        }
    }
    __syncthreads();
    // 2. expert offsets
    block_exclusive_scan(s_kept, s_off, E, s_warp);
    const int total = s_off[E];
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= E; e += kScanThreads) a.o.offsets[e] = s_off[e];
        if (threadIdx.x == 0) *a.o.n_dropped = n - total;
        if (a.o.p_part && E <= kWarpColumnMaxE) {
            // load statistics: f = counts/(T k), p = mean softmax row, L = alpha E sum f p
            // (p: the column-sum order moe_load_stats uses; L: terms added in expert order)
            s_red[threadIdx.x] = 0.f;
            __syncthreads();
            for (int e = warp; e < E; e += kScanWarps) {
                const float ps = warp_column_sum(a.o.p_part, a.o.p_nblk, E, e);
                if (lane == 0) {
                    const float pm = ps / (float)a.T;
                    const float f = (float)s_wcnt[e] / ((float)a.T * (float)a.k);
                    if (a.o.p_mean) a.o.p_mean[e] = pm;
                    if (a.o.f) a.o.f[e] = f;
                    s_red[e] = f * pm;
                }
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                float acc = 0.f;
                for (int i = 0; i < kScanThreads; ++i) acc += s_red[i];
                if (a.o.L) *a.o.L = a.o.alpha * (float)E * acc;
            }
        } else if (a.o.p_part) {
            // load statistics: f = counts/(T k), p = mean softmax row, L = alpha E sum f p
            float* s_p = reinterpret_cast<float*>(s_pb + kScanWarps * E);  // [p_nblk][E] when staged
            if (a.p_stage) {
                const int n = a.o.p_nblk * E;
#pragma unroll 16
                for (int i = threadIdx.x; i < n; i += kScanThreads) s_p[i] = __ldg(a.o.p_part + i);
                __syncthreads();
            }
            float part = 0.f;
            for (int e = threadIdx.x; e < E; e += kScanThreads) {
                float ps = 0.f;  // row order, as moe_load_stats sums it; 32 loads in flight
                if (a.p_stage) {
                    for (int b = 0; b < a.o.p_nblk; ++b) ps += s_p[b * E + e];
                } else {
                    for (int b0 = 0; b0 < a.o.p_nblk; b0 += 32) {
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            v[j] = b0 + j < a.o.p_nblk ? __ldg(a.o.p_part + (size_t)(b0 + j) * E + e) : 0.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (b0 + j < a.o.p_nblk) ps += v[j];
                    }
                }
                const float pm = ps / (float)a.T;
                const float f = (float)s_wcnt[e] / ((float)a.T * (float)a.k);
                if (a.o.p_mean) a.o.p_mean[e] = pm;
                if (a.o.f) a.o.f[e] = f;
                part += f * pm;
            }
            s_red[threadIdx.x] = part;
            __syncthreads();
            if (threadIdx.x == 0) {
                float acc = 0.f;
                for (int i = 0; i < kScanThreads; ++i) acc += s_red[i];
                if (a.o.L) *a.o.L = a.o.alpha * (float)E * acc;
            }
        }
    }
    // positions past the kept total: sorted_token_ids = -1, gates_perm = 0
    for (int pos = total + blockIdx.x * kScanThreads + threadIdx.x; pos < n; pos += gridDim.x * kScanThreads) {
        a.o.sorted_token_ids[pos] = -1;
        a.o.gates_perm[pos] = 0.f;
    }
    __syncthreads();

    // 3. stable ranks: warp w owns a contiguous sub-range of this block's entries
    const int lo = blockIdx.x * a.chunk * a.k;
    const int hi = min(n, lo + a.chunk * a.k);
    const int per_warp = (hi - lo + kScanWarps - 1) / kScanWarps;
    const int wlo = min(hi, lo + warp * per_warp);
    const int whi = min(hi, wlo + per_warp);
    int* wcnt = s_wcnt + warp * E;
    for (int e = lane; e < E; e += 32) wcnt[e] = 0;
    __syncwarp();
    for (int base = wlo; base < whi; base += 32) {  // pass A: per-warp counts
        const int i = base + lane;
        int e = (i < whi) ? a.ids[i] : -1;
        if (e >= E) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e < 0 ? -1 - lane : e);
        if (e >= 0 && lane == __ffs(peers) - 1) wcnt[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kScanThreads) {  // per-warp starting ranks
        int run = s_before[e];
        for (int w = 0; w < kScanWarps; ++w) {
            const int c = s_wcnt[w * E + e];
            s_wcnt[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int base = wlo; base < whi; base += 32) {  // pass B: ranks and positions
        const int i = base + lane;
        int e = (i < whi) ? a.ids[i] : -1;
        if (e >= E || (i < whi && e < 0)) {
            record_status(a.status, kStatusBounds);
            e = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e < 0 ? -1 - lane : e);
        int rank = 0;
        if (e >= 0) rank = wcnt[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) wcnt[e] += __popc(peers);
        __syncwarp();
        if (i < whi) {
            int pos = -1;
            if (e >= 0 && (a.capacity < 0 || rank < a.capacity)) pos = s_off[e] + rank;
            if (pos >= 0 && pos >= s_off[e + 1]) {  // ids that disagree with the histogram rows
                record_status(a.status, kStatusBounds);
                pos = -1;
            }
            a.o.slot_pos[i] = pos;
            if (pos >= 0) {
                a.o.sorted_token_ids[pos] = i / a.k;
                a.o.gates_perm[pos] = a.gates[i];
            }
        }
    }
    __syncthreads();
    pdl_trigger();
}

template <typename T>
__global__ void __launch_bounds__(256) gather_rows_kernel(int Tn, int d, const int32_t* __restrict__ offsets_end,
                                                          const int32_t* __restrict__ sorted_token_ids,
                                                          const T* __restrict__ x, T* __restrict__ x_perm,
                                                          int rows_max, int* status) {
    pdl_wait();
    const int total = min(*offsets_end, rows_max);
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int vec = 16 / sizeof(T);
    for (int row = warp; row < total; row += nwarps) {
        const int t = sorted_token_ids[row];
        if (t < 0 || t >= Tn) {
            if (lane == 0) record_status(status, kStatusBounds);
            continue;
        }
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)row * d);
        for (int c = lane; c < d / vec; c += 32) dst[c] = __ldg(src + c);
    }
    __syncthreads();
    pdl_trigger();
}

}  // namespace

cudaError_t launch_group_hist(int T, int E, int k, int chunk, const int32_t* topk_ids, int32_t* block_hist,
                              int* status, cudaStream_t s) {
    const int nblk = (T + chunk - 1) / chunk;
    if (nblk == 0) return cudaSuccess;
    launch_pdl(group_hist_kernel, dim3(nblk), dim3(kRouterThreads), E * sizeof(int), s, T, E, k, chunk, topk_ids, block_hist, status);
    return cudaGetLastError();
}

cudaError_t launch_group_scan(int T, int E, int k, int chunk, int capacity, const int32_t* topk_ids,
                              const float* gates, const int32_t* block_hist, const GroupOut& o, int* status,
                              cudaStream_t s) {
    const int nblk = (T + chunk - 1) / chunk;
    if (nblk == 0) return cudaSuccess;
    const int p_stage = o.p_part && E > kWarpColumnMaxE && (long long)o.p_nblk * E <= kScanStageFloats ? 1 : 0;
    ScanArgs a{T, E, k, chunk, capacity, nblk, p_stage, topk_ids, gates, block_hist, o, status};
    const size_t smem = sizeof(int) * ((size_t)3 * E + 1 + (size_t)kScanWarps * E + kScanWarps + 1) +
                        sizeof(float) * kScanThreads + sizeof(int) * (size_t)kScanWarps * E +
                        (p_stage ? sizeof(float) * (size_t)o.p_nblk * E : 0);
    if (smem > 48 * 1024)  // (at most 78 KB for the largest E the library takes, 64 KB more when staging p)
        cudaFuncSetAttribute(group_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_pdl(group_scan_kernel, dim3(nblk), dim3(kScanThreads), smem, s, a);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(int dtype, int T, int d, int rows_max, const int32_t* offsets_end,
                               const int32_t* sorted_token_ids, const void* x, void* x_perm, int* status,
                               cudaStream_t s) {
    if (rows_max == 0) return cudaSuccess;
    // SM count of the current device, remembered per device ordinal
    static int sms_of[64] = {0};
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && sms_of[dev] > 0) {
        sms = sms_of[dev];
    } else if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && dev >= 0 &&
               dev < 64) {
        sms_of[dev] = sms;
    }
    const int want = (rows_max + 7) / 8;  // 8 warps per block, one row per warp
    const int grid = want < sms * 8 ? want : sms * 8;
    if (dtype == MOE_BF16)
        launch_pdl(gather_rows_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s, T, d, offsets_end, sorted_token_ids,
                                                               static_cast<const __nv_bfloat16*>(x),
                                                               static_cast<__nv_bfloat16*>(x_perm), rows_max, status);
    else
        launch_pdl(gather_rows_kernel<float>, dim3(grid), dim3(256), 0, s, T, d, offsets_end, sorted_token_ids,
                                                       static_cast<const float*>(x), static_cast<float*>(x_perm),
                                                       rows_max, status);
    return cudaGetLastError();
}

}  // namespace moe
