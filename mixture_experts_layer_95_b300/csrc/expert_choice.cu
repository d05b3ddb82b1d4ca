// expert_choice.cu -- expert-choice routing: every expert picks its tokens.
//
// "One Deep Concept #04", section 11 "Expert Choice -- Reverse Who Selects
// Whom": instead of each token choosing its experts, each expert chooses a
// fixed-size bucket of C tokens, so every expert's load is exactly C while a
// token may receive any number of experts (none included).  Scores are the
// router's softmax probabilities p[t][e] (written by the router kernels); the
// gate of a chosen (t, e) is p[t][e], not renormalised.
//
// ec_select_kernel: one 1024-thread block per expert.
//  1. Radix select of the C-th largest score: fp32 probabilities are >= 0, so
//     their bit patterns order like their values; four 8-bit passes of a
//     shared-memory histogram over the tokens still matching the prefix found
//     so far give the exact threshold key K and how many tokens equal to K
//     still belong in the bucket.
//  2. One sweep over the tokens in index order, 1024 at a time: a block-wide
//     ballot scan ranks the ties (key == K) so that the lowest token indices
//     win, a second scan gives each chosen token its position, and the bucket
//     is written in ascending token order -- segment e of the permuted rows
//     is rows [e*C, (e+1)*C).  The block also writes column e of the [T][E]
//     slot map (row or -1) that the combine reads.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kEcThreads = 1024;
constexpr int kEcWarps = kEcThreads / 32;  // 32: one scan lane per warp
static_assert(kEcWarps == 32, "the block scan below assumes 32 warps");

// Exclusive block-wide count of `flag` over threads 0..threadIdx.x-1 (in
// thread order); `total` receives the block's count.  s_scan: 64 ints.
__device__ __forceinline__ int block_flag_scan(bool flag, int* s_scan, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned b = __ballot_sync(0xffffffffu, flag);
    if (lane == 0) s_scan[warp] = __popc(b);
    __syncthreads();
    if (warp == 0) {
        int v = s_scan[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        s_scan[32 + lane] = v;  // inclusive
    }
    __syncthreads();
    total = s_scan[63];
    const int r = (warp ? s_scan[32 + warp - 1] : 0) + __popc(b & ((1u << lane) - 1u));
    __syncthreads();  // s_scan is reused by the next call
    return r;
}

__global__ void __launch_bounds__(kEcThreads) ec_select_kernel(int Tn, int E, int C, const float* __restrict__ probs,
                                                               int32_t* __restrict__ sorted_token_ids,
                                                               float* __restrict__ gates_perm,
                                                               int32_t* __restrict__ slot_pos,
                                                               int32_t* __restrict__ counts,
                                                               int32_t* __restrict__ kept,
                                                               int32_t* __restrict__ offsets,
                                                               int32_t* __restrict__ n_empty) {
    pdl_wait();
    __shared__ int s_hist[256];
    __shared__ int s_scan[64];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;
    const int e = blockIdx.x;
    const float* col = probs + e;  // p[t][e] at col[t * E]

    // 1: the C-th largest key, 8 bits at a time from the top
    uint32_t prefix = 0, mask = 0;
    int need = C;  // tokens still to take among those matching `prefix`
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kEcThreads) s_hist[i] = 0;
        __syncthreads();
        for (int t = threadIdx.x; t < Tn; t += kEcThreads) {
            const uint32_t key = __float_as_uint(__ldg(col + (size_t)t * E));
            if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int above = 0, b = 255;
            for (; b > 0; --b) {
                if (above + s_hist[b] >= need) break;
                above += s_hist[b];
            }
            s_prefix = prefix | ((uint32_t)b << shift);
            s_need = need - above;
        }
        __syncthreads();
        prefix = s_prefix;
        need = s_need;
        mask |= 255u << shift;
    }
    const uint32_t K = prefix;  // all C chosen keys are > K, or == K and among the first `need` ties

    // 2: ascending token order; ties to the lower token index
    int run_eq = 0, run_take = 0;
    for (int base = 0; base < Tn; base += kEcThreads) {
        const int t = base + threadIdx.x;
        const bool valid = t < Tn;
        const float p = valid ? __ldg(col + (size_t)t * E) : 0.f;
        const uint32_t key = __float_as_uint(p);
        const bool eq = valid && key == K;
        int eq_total, take_total;
        const int eq_rank = run_eq + block_flag_scan(eq, s_scan, eq_total);
        const bool take = valid && (key > K || (eq && eq_rank < need));
        const int pos = run_take + block_flag_scan(take, s_scan, take_total);
        if (valid) {
            const bool in = take && pos < C;  // exactly C are taken; pos < C only guards the writes
            const int row = e * C + pos;
            slot_pos[(size_t)t * E + e] = in ? row : -1;
            if (in) {
                sorted_token_ids[row] = t;
                gates_perm[row] = p;
            }
        }
        run_eq += eq_total;
        run_take += take_total;
    }
    if (threadIdx.x == 0) {
        if (counts) counts[e] = C;
        if (kept) kept[e] = C;
        offsets[e + 1] = (e + 1) * C;
        if (e == 0) {
            offsets[0] = 0;
            if (n_empty) *n_empty = 0;  // counted afterwards by the combine
        }
    }
    __syncthreads();
    pdl_trigger();
}

}  // namespace

cudaError_t launch_ec_select(int T, int E, int C, const float* probs, int32_t* sorted_token_ids, float* gates_perm,
                             int32_t* slot_pos, int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* n_empty,
                             cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    launch_pdl(ec_select_kernel, dim3(E), dim3(kEcThreads), 0, s, T, E, C, probs, sorted_token_ids, gates_perm,
               slot_pos, counts, kept, offsets, n_empty);
    return cudaGetLastError();
}

}  // namespace moe
