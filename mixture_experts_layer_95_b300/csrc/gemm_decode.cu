// gemm_decode.cu -- grouped expert GEMMs for decode-sized batches, with the
// expert weights on the M side of the tensor-core MMA.
//
// The same two problems as gemm_tc.cu ("Mixture of experts (MoE)" handbook,
// grouped by expert; its SwiGLU Expert, down(silu(gate(x)) * up(x))):
//   up:   H[r, :] = silu(X[r] W1_g^T) * (X[r] W3_g^T)
//   down: Y[r, :] = gate[r] * (H[r] W2_g^T)
// but for batches with a few rows per expert, where the layer is bound by
// streaming the touched experts' weights from HBM.  A 128-row token tile
// would waste most of every stage on absent rows, so the operands swap:
// 128-row slices of the weight tile are the MMA's A operand (M = 128 weight
// rows, one TMEM lane each) and NT token rows its B operand (N = NT), i.e.
// D^T = W X^T.  A stage then holds a 256-row weight tile (32 KB in bf16, 16 KB
// as FP8 codes) plus NT token rows (NT * 128 bytes), so 5 to 7 stages -- 160
// KB of bf16 or 112 KB of FP8 weights -- stay in flight per SM.  The epilogue
// runs along the weight-row axis: the 32 lanes of a warp hold 32 consecutive
// output columns, so every store of one token row is one contiguous segment.
//
// Roles: warp 0 TMA producer (weight tile + token rows, gathered with
// tile::gather4 when the rows come straight from the token matrix); warp 1
// TMEM allocation and the single MMA-issuing thread (two M=128 MMAs per
// K=16 step, one per half of the weight tile); warps 2-5 epilogue; with FP8
// weights, warps 6-13 widen each one-byte weight tile into a bf16 tile (two
// buffers) before the MMA reads it.  Split-K, per-row gates, FP8 per-channel
// scales and the bounded mbarrier waits are as in gemm_tc.cu.
#include <stdlib.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {
using namespace tc;

constexpr int WR = 256;                  // weight rows per tile (SwiGLU: 128 of W1 + 128 of W3)
constexpr int WB16 = WR * BK * 2;        // bf16 weight tile bytes (one k-block of 64)
// A stage carries KPS k-blocks: 1 for bf16 weights; 2 for FP8, so that every
// weight row of a stage is 128 contiguous bytes, as for bf16 (a 64-byte row
// per TMA request halves the bytes each request brings in).
template <bool W8>
constexpr int kps() {
    return W8 ? 2 : 1;
}
constexpr int DEC_THREADS = 192;         // producer, MMA, 4 epilogue warps
constexpr int DEC_W8_THREADS = 192 + 256;  // + 8 widening warps
constexpr int DEC_WIDE = 2;              // widened bf16 weight tiles (FP8)
constexpr int DEC_MAX_RING = 8;
constexpr int DEC_TMEM_COLS = 256;       // two accumulators of 2 x NT columns (NT <= 64)
constexpr int MAX_GROUPS = kMaxExperts;

struct DecParams {  // CUtensorMap members carry their own 64-byte alignment
    CUtensorMap tmX[2];   // token rows: a gather map (one-row box) or a tile map (NT-row box)
    CUtensorMap tmW1[2];  // weights: W1 (SwiGLU) or W2 (down)
    CUtensorMap tmW2[2];  // W3 (SwiGLU)
    const int32_t* offsets[2];
    void* out[2];
    const float* row_scale[2];
    const float* wscale1[2];
    const float* wscale2[2];
    const int32_t* x_gather[2];
    int G[2], M[2], N[2], K[2], x_rows[2], x_src_rows[2];
    float* part[2];
    int part_cols[2];
    int nprob, ksplit;
    int* status;
    uint64_t wait_limit_ns;
    int stall_producer;
};

struct DecTail {
    uint64_t full[DEC_MAX_RING];
    uint64_t empty[DEC_MAX_RING];
    uint64_t wfull[DEC_WIDE];
    uint64_t wempty[DEC_WIDE];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint32_t tmem_base;
    int abort_flag;
    int total[2];
    int gbase[2];
    int tile_start[MAX_GROUPS + 1];
    int row0[MAX_GROUPS + 1];
    int rows[MAX_GROUPS + 1];
};

constexpr int kSmemLimit = 232448;  // 227 KB opt-in per CTA

template <bool W8, int NT>
constexpr int dec_slot_bytes() {
    return WR * 128 + kps<W8>() * NT * BK * 2;  // 256 weight rows x 128 bytes, then KPS token tiles
}

template <bool W8, int NT>
constexpr int dec_stages() {
    return (kSmemLimit - 1024 - (int)sizeof(DecTail) - (W8 ? DEC_WIDE * WB16 : 0)) / dec_slot_bytes<W8, NT>() >
                   DEC_MAX_RING
               ? DEC_MAX_RING
               : (kSmemLimit - 1024 - (int)sizeof(DecTail) - (W8 ? DEC_WIDE * WB16 : 0)) / dec_slot_bytes<W8, NT>();
}

template <bool W8, int NT>
constexpr size_t dec_smem_bytes() {
    return 1024 + (size_t)dec_stages<W8, NT>() * dec_slot_bytes<W8, NT>() + (W8 ? (size_t)DEC_WIDE * WB16 : 0) +
           sizeof(DecTail);
}

static_assert(dec_stages<false, 32>() >= 4 && dec_stages<false, 64>() >= 4, "bf16 decode ring too shallow");
static_assert(dec_stages<true, 32>() >= 3 && dec_stages<true, 64>() >= 3, "FP8 decode ring too shallow");
static_assert(dec_smem_bytes<true, 32>() <= kSmemLimit && dec_smem_bytes<false, 64>() <= kSmemLimit &&
                  dec_smem_bytes<true, 64>() <= kSmemLimit && dec_smem_bytes<false, 32>() <= kSmemLimit,
              "decode GEMM exceeds shared memory");

struct DTile {
    int prob, g, m, n;
    int x_row0, rows_valid;
    int ks, kb0, kb1;  // K slice and its range of stages [kb0, kb1) (KPS k-blocks each)
};

// output columns one tile covers: 128 (the W1/W3 pair) or 256 (W2)
template <int MODE>
__device__ __forceinline__ int dec_cols() {
    return MODE == kGemmSwiGLU ? WR / 2 : WR;
}

template <int MODE, int NT, int KPS>
__device__ __forceinline__ DTile dec_tile(const DecTail& st, const DecParams& p, int id) {
    DTile t;
    t.prob = (id < st.total[0]) ? 0 : 1;
    const int local = id - (t.prob ? st.total[0] : 0);
    const int gb = st.gbase[t.prob];
    const int* ts = st.tile_start + gb;
    int lo = 0, hi = p.G[t.prob] - 1;  // largest g with ts[g] <= local
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ts[mid] <= local) lo = mid;
        else hi = mid - 1;
    }
    t.g = lo;
    const int rows = st.rows[gb + lo];
    const int mt = (rows + NT - 1) / NT;
    int r = local - ts[lo];
    t.ks = r % p.ksplit;  // K slices of one output tile are adjacent, then token chunks
    r /= p.ksplit;
    t.n = r / mt;
    t.m = r - t.n * mt;
    t.x_row0 = st.row0[gb + lo] + t.m * NT;
    t.rows_valid = min(NT, rows - t.m * NT);
    const int nk = (p.K[t.prob] + KPS * BK - 1) / (KPS * BK);
    t.kb0 = t.ks * nk / p.ksplit;
    t.kb1 = (t.ks + 1) * nk / p.ksplit;
    return t;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

// Widening of one k-block (64 codes) of an FP8 stage whose weight rows are
// 128 bytes apart, by `nthreads` threads (the converter warps), into a bf16
// K-major 128-byte-swizzled tile; layout as widen_b_tile in tc_ptx.cuh.
__device__ __forceinline__ void widen_tile(const uint8_t* src, uint8_t* dst, int tid, int nthreads) {
#pragma unroll
    for (int idx = tid; idx < WR * 8; idx += nthreads) {
        const int r = idx >> 3, c = idx & 7;
        const uint2 raw = *reinterpret_cast<const uint2*>(src + r * 128 + c * 8);
        uint4 out;
        out.x = e4m3x2_to_bf16x2(__byte_perm(raw.x, 0u, 0x1404));
        out.y = e4m3x2_to_bf16x2(__byte_perm(raw.x, 0u, 0x3424));
        out.z = e4m3x2_to_bf16x2(__byte_perm(raw.y, 0u, 0x1404));
        out.w = e4m3x2_to_bf16x2(__byte_perm(raw.y, 0u, 0x3424));
        *reinterpret_cast<uint4*>(dst + r * (BK * 2) + ((c ^ (r & 7)) << 4)) = out;
    }
}

// Epilogue of one tile for this thread's weight row.  The accumulator half h
// (TMEM columns h*NT .. h*NT+NT-1) holds, per token column j, the dot product
// of token row x_row0 + j with weight row  (tile row h*128 + lane).
template <int MODE, int NT>
__device__ __forceinline__ void dec_epilogue(const DecParams& p, const DTile& t, uint32_t tacc, int wrow) {
    const int N = p.N[t.prob];
    const size_t gN = static_cast<size_t>(t.g) * N;
    if (MODE == kGemmSwiGLU) {
        const int f = t.n * (WR / 2) + wrow;  // output column (hidden channel)
        const bool live = f < N;
        const float s1 = (live && p.wscale1[t.prob]) ? __ldg(p.wscale1[t.prob] + gN + f) : 1.0f;
        const float s3 = (live && p.wscale2[t.prob]) ? __ldg(p.wscale2[t.prob] + gN + f) : 1.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < NT; c0 += 32) {
            uint32_t g[32], u[32];
            __syncwarp();
            tmem_ld32(tacc + c0, g);
            tmem_ld32(tacc + NT + c0, u);
            tmem_ld_wait();
            if (!live) continue;
            const int jn = min(32, t.rows_valid - c0);
            if (p.ksplit > 1) {
                const size_t pc = static_cast<size_t>(p.part_cols[t.prob]);
                float* base = p.part[t.prob] + (static_cast<size_t>(t.ks) * p.x_rows[t.prob] + t.x_row0 + c0) * pc;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < jn) {
                        base[j * pc + f] = s1 * __uint_as_float(g[j]);
                        base[j * pc + N + f] = s3 * __uint_as_float(u[j]);
                    }
            } else {
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[t.prob]) + (size_t)(t.x_row0 + c0) * N + f;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < jn)
                        out[(size_t)j * N] =
                            __float2bfloat16_rn(silu_mul(s1 * __uint_as_float(g[j]), s3 * __uint_as_float(u[j])));
            }
        }
    } else {
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            const int o = t.n * WR + h * 128 + wrow;  // output column
            const bool live = o < N;
            const float ws = (live && p.wscale1[t.prob]) ? __ldg(p.wscale1[t.prob] + gN + o) : 1.0f;
#pragma unroll 1
            for (int c0 = 0; c0 < NT; c0 += 32) {
                uint32_t v[32];
                __syncwarp();
                tmem_ld32(tacc + h * NT + c0, v);
                tmem_ld_wait();
                if (!live) continue;
                const int jn = min(32, t.rows_valid - c0);
                const size_t row = (size_t)(t.x_row0 + c0);
                const float* rs = p.row_scale[t.prob] ? p.row_scale[t.prob] + row : nullptr;
                float* dst = p.ksplit > 1
                                 ? p.part[t.prob] + (static_cast<size_t>(t.ks) * p.x_rows[t.prob] + row) * N + o
                                 : static_cast<float*>(p.out[t.prob]) + row * N + o;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < jn) dst[(size_t)j * N] = (rs ? __ldg(rs + j) : 1.0f) * ws * __uint_as_float(v[j]);
            }
        }
    }
}

template <int MODE, bool W8, int NT>
__global__ void __launch_bounds__(W8 ? DEC_W8_THREADS : DEC_THREADS, 1)
    grouped_gemm_decode_kernel(const __grid_constant__ DecParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int NST = dec_stages<W8, NT>();
    constexpr int SLOT = dec_slot_bytes<W8, NT>();
    constexpr int KPS = kps<W8>();
    constexpr int WBYTES = WR * 128;   // weight bytes at the start of a stage; KPS token tiles follow
    constexpr int XBYTES = NT * BK * 2;  // one token tile
    static_assert(MODE == kGemmSwiGLU || MODE == kGemmScale, "decode GEMM: SwiGLU and Scale modes");
    uint8_t* wide = smem + (size_t)NST * SLOT;  // FP8: widened weight tiles
    DecTail& st = *reinterpret_cast<DecTail*>(wide + (W8 ? (size_t)DEC_WIDE * WB16 : 0));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &st.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&st.full[s], 1);
            mbar_init(&st.empty[s], 1);
        }
        for (int w = 0; w < DEC_WIDE; ++w) {
            mbar_init(&st.wfull[w], 8);  // one arrival per widening warp
            mbar_init(&st.wempty[w], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&st.tmem_full[a], 1);
            mbar_init(&st.tmem_empty[a], 4);
        }
        st.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        for (int q = 0; q < p.nprob; ++q) {
            prefetch_tmap(&p.tmX[q]);
            prefetch_tmap(&p.tmW1[q]);
            if (MODE == kGemmSwiGLU) prefetch_tmap(&p.tmW2[q]);
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&st.tmem_base)),
                     "r"(DEC_TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    pdl_wait();
    if (warp == 2) {
        for (int q = 0; q < 2; ++q) {
            int carry = 0;
            const int gb = q == 0 ? 0 : p.G[0];
            if (lane == 0) st.gbase[q] = gb;
            if (q < p.nprob) {
                const int ncb = (p.N[q] + dec_cols<MODE>() - 1) / dec_cols<MODE>();
                for (int base = 0; base < p.G[q]; base += 32) {
                    const int g = base + lane;
                    int tiles = 0;
                    if (g < p.G[q]) {
                        int lo = 0, hi = p.M[q];
                        if (p.offsets[q]) {
                            lo = p.offsets[q][g];
                            hi = p.offsets[q][g + 1];
                        }
                        if (lo < 0 || hi < lo || hi > p.x_rows[q]) {
                            record_status(p.status, kStatusBounds);
                            lo = hi = 0;
                        }
                        st.row0[gb + g] = lo;
                        st.rows[gb + g] = hi - lo;
                        tiles = ((hi - lo + NT - 1) / NT) * ncb * p.ksplit;
                    }
                    int incl = tiles;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += y;
                    }
                    if (g < p.G[q]) st.tile_start[gb + g] = carry + incl - tiles;
                    carry += __shfl_sync(0xffffffffu, incl, 31);
                }
            }
            if (lane == 0) st.total[q] = carry;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = st.tmem_base;
    const int total_tiles = st.total[0] + st.total[1];

    if (warp == 0) {
        // ---------------- TMA producer: weight tile + token rows per k-block ----------------
        int s = 0;
        uint32_t ph = 0;
        uint32_t issued_parity[NST];
        bool used[NST];
        for (int i = 0; i < NST; ++i) used[i] = false;
        bool dead = p.stall_producer != 0;
        for (int id = blockIdx.x; id < total_tiles && !dead; id += gridDim.x) {
            const DTile t = dec_tile<MODE, NT, KPS>(st, p, id);
            const int w_row0 = t.g * p.N[t.prob] + t.n * dec_cols<MODE>();
            const int32_t* gidx = p.x_gather[t.prob];
            int rows4[4] = {0, 0, 0, 0};
            if (gidx) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = lane * 4 + i;
                    int v = r < t.rows_valid ? __ldg(gidx + t.x_row0 + r) : 0;
                    if (v < 0 || v >= p.x_src_rows[t.prob]) {
                        if (r < t.rows_valid) record_status(p.status, kStatusBounds);
                        v = 0;
                    }
                    rows4[i] = v;
                }
            }
            for (int kb = t.kb0; kb < t.kb1; ++kb) {
                if (!mbar_wait(&st.empty[s], ph ^ 1u, abort_flag, p.status, p.wait_limit_ns)) {
                    dead = true;
                    break;
                }
                uint8_t* sw = smem + (size_t)s * SLOT;
                uint8_t* sx = sw + WBYTES;
                if (lane == 0) {
                    const uint32_t x_bytes =
                        gidx ? (uint32_t)((t.rows_valid + 3) / 4) * 4 * (BK * 2) : (uint32_t)XBYTES;
                    mbar_expect_tx(&st.full[s], WBYTES + KPS * x_bytes);
                    // weight columns of this stage: KPS * 64 elements (bf16: 64, FP8: 128 bytes)
                    const int wc = kb * KPS * BK;
                    if (MODE == kGemmSwiGLU) {
                        tma_load_2d(sw, &p.tmW1[t.prob], wc, w_row0, &st.full[s]);
                        tma_load_2d(sw + WBYTES / 2, &p.tmW2[t.prob], wc, w_row0, &st.full[s]);
                    } else {
                        tma_load_2d(sw, &p.tmW1[t.prob], wc, w_row0, &st.full[s]);
                    }
                    if (!gidx)
                        for (int h = 0; h < KPS; ++h)
                            tma_load_2d(sx + h * XBYTES, &p.tmX[t.prob], (kb * KPS + h) * BK, t.x_row0, &st.full[s]);
                }
                if (gidx && lane * 4 < t.rows_valid)
                    for (int h = 0; h < KPS; ++h)
                        tma_gather4(sx + h * XBYTES + lane * 4 * (BK * 2), &p.tmX[t.prob], (kb * KPS + h) * BK,
                                    rows4[0], rows4[1], rows4[2], rows4[3], &st.full[s]);
                issued_parity[s] = ph;
                used[s] = true;
                if (++s == NST) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            volatile int no_abort = 0;
            for (int i = 0; i < NST; ++i)
                if (used[i]) mbar_wait(&st.full[i], issued_parity[i], &no_abort, nullptr, kDrainLimitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, NT);
            int s = 0, w = 0;
            uint32_t ph = 0, pw = 0;
            int it = 0;
            bool dead = false;
            for (int id = blockIdx.x; id < total_tiles && !dead; id += gridDim.x, ++it) {
                const DTile t = dec_tile<MODE, NT, KPS>(st, p, id);
                const int acc = it & 1;
                const uint32_t use = static_cast<uint32_t>(it >> 1);
                if (!mbar_wait(&st.tmem_empty[acc], (use & 1u) ^ 1u, abort_flag, p.status, p.wait_limit_ns)) break;
                tc_fence_after();
                const uint32_t dtm = tmem_base + static_cast<uint32_t>(acc * 2 * NT);
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait(&st.full[s], ph, abort_flag, p.status, p.wait_limit_ns)) {
                        dead = true;
                        break;
                    }
                    for (int h = 0; h < KPS && !dead; ++h) {
                        if (W8 && !mbar_wait(&st.wfull[w], pw, abort_flag, p.status, p.wait_limit_ns)) {
                            dead = true;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sw =
                            W8 ? smem_u32(wide + (size_t)w * WB16) : smem_u32(smem + (size_t)s * SLOT);
                        const uint32_t sx = smem_u32(smem + (size_t)s * SLOT + WBYTES + h * XBYTES);
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            const uint64_t xdesc = sdesc_k_sw128(sx + kk * UMMA_K * 2);
                            const uint32_t accf = (kb != t.kb0 || h != 0 || kk != 0) ? 1u : 0u;
                            umma_bf16(dtm, sdesc_k_sw128(sw + kk * UMMA_K * 2), xdesc, idesc, accf);
                            umma_bf16(dtm + NT, sdesc_k_sw128(sw + 128 * BK * 2 + kk * UMMA_K * 2), xdesc, idesc,
                                      accf);
                        }
                        if (W8) {
                            umma_commit(&st.wempty[w]);
                            if (++w == DEC_WIDE) {
                                w = 0;
                                pw ^= 1u;
                            }
                        }
                    }
                    if (dead) break;
                    umma_commit(&st.empty[s]);
                    if (++s == NST) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (dead) break;
                umma_commit(&st.tmem_full[acc]);
            }
        }
    } else if (warp < 6) {
        // ---------------- epilogue (warps 2..5): one weight row per thread ----------------
        const int quarter = warp & 3;
        const int wrow = quarter * 32 + lane;
        int it = 0;
        for (int id = blockIdx.x; id < total_tiles; id += gridDim.x, ++it) {
            const DTile t = dec_tile<MODE, NT, KPS>(st, p, id);
            const int acc = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            if (!mbar_wait(&st.tmem_full[acc], use & 1u, abort_flag, p.status, p.wait_limit_ns)) break;
            tc_fence_after();
            const uint32_t tacc =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * 2 * NT);
            dec_epilogue<MODE, NT>(p, t, tacc, wrow);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&st.tmem_empty[acc]);
        }
    } else if constexpr (W8) {
        // ---------------- widening warps (6..13), FP8 weights ----------------
        const int ctid = threadIdx.x - DEC_THREADS;  // 0..255
        int s = 0, w = 0;
        uint32_t ph = 0, pw = 0;
        bool dead = false;
        for (int id = blockIdx.x; id < total_tiles && !dead; id += gridDim.x) {
            const DTile t = dec_tile<MODE, NT, KPS>(st, p, id);
            for (int kb = t.kb0; kb < t.kb1; ++kb) {
                const bool ok_raw = mbar_wait(&st.full[s], ph, abort_flag, p.status, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok_raw)) {
                    dead = true;
                    break;
                }
                for (int h = 0; h < KPS; ++h) {
                    const bool ok_w = mbar_wait(&st.wempty[w], pw ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                    if (!__all_sync(0xffffffffu, ok_w)) {
                        dead = true;
                        break;
                    }
                    widen_tile(smem + (size_t)s * SLOT + h * BK, wide + (size_t)w * WB16, ctid,
                               DEC_W8_THREADS - DEC_THREADS);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&st.wfull[w]);
                    if (++w == DEC_WIDE) {
                        w = 0;
                        pw ^= 1u;
                    }
                }
                if (dead) break;
                if (++s == NST) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {
        }
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(DEC_TMEM_COLS));
    }
    pdl_trigger();
}

template <int MODE, bool W8, int NT>
cudaError_t launch_dec(const DecParams& prm, int grid, cudaStream_t s) {
    static uint64_t attr_set_mask = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (!bit || !(attr_set_mask & bit)) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_decode_kernel<MODE, W8, NT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(dec_smem_bytes<W8, NT>()));
        if (e != cudaSuccess) return e;
        attr_set_mask |= bit;
    }
    launch_pdl(grouped_gemm_decode_kernel<MODE, W8, NT>, dim3(grid), dim3(W8 ? DEC_W8_THREADS : DEC_THREADS),
               dec_smem_bytes<W8, NT>(), s, prm);
    return cudaGetLastError();
}

template <int MODE, bool W8>
cudaError_t launch_dec_nt(const DecParams& prm, int nt, int grid, cudaStream_t s) {
    return nt == 32 ? launch_dec<MODE, W8, 32>(prm, grid, s) : launch_dec<MODE, W8, 64>(prm, grid, s);
}

}  // namespace

cudaError_t launch_gemm_decode(int mode, const GemmProblem* probs, int nprob, int* status, int num_sms,
                               cudaStream_t s, int ksplit, bool w8, int nt) {
    if (nprob < 1 || nprob > 2 || ksplit < 1 || (nt != 32 && nt != 64)) return cudaErrorInvalidValue;
    if (mode != kGemmSwiGLU && mode != kGemmScale) return cudaErrorInvalidValue;
    DecParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.ksplit = ksplit;
    const int w_box = mode == kGemmSwiGLU ? WR / 2 : WR;
    if (probs[0].G + (nprob > 1 ? probs[1].G : 0) > MAX_GROUPS + 1) return cudaErrorInvalidValue;
    for (int q = 0; q < nprob; ++q) {
        const GemmProblem& g = probs[q];
        if (g.G < 1 || g.G > MAX_GROUPS || g.out2 || g.A2) return cudaErrorInvalidValue;
        if (w8 && (g.K % 16 != 0 || !g.wscale1 || (mode == kGemmSwiGLU && !g.wscale2))) return cudaErrorInvalidValue;
        if (g.a_gather) {
            if (!make_tmap(&prm.tmX[q], g.A, g.a_src_rows, g.K, 1)) return cudaErrorInvalidValue;
            prm.x_gather[q] = g.a_gather;
            prm.x_src_rows[q] = g.a_src_rows;
        } else if (!make_tmap(&prm.tmX[q], g.A, g.a_rows, g.K, nt)) {
            return cudaErrorInvalidValue;
        }
        // FP8 stages hold 128 codes (two k-blocks) of every weight row
        const bool ok1 = w8 ? make_tmap_u8(&prm.tmW1[q], g.B1, g.G * g.N, g.K, w_box, 2 * BK)
                            : make_tmap(&prm.tmW1[q], g.B1, g.G * g.N, g.K, w_box);
        if (!ok1) return cudaErrorInvalidValue;
        if (mode == kGemmSwiGLU) {
            const bool ok2 = w8 ? make_tmap_u8(&prm.tmW2[q], g.B2, g.G * g.N, g.K, w_box, 2 * BK)
                                : make_tmap(&prm.tmW2[q], g.B2, g.G * g.N, g.K, w_box);
            if (!ok2) return cudaErrorInvalidValue;
        }
        if (ksplit > 1) {
            const int kstep = (w8 ? 2 : 1) * BK;
            if (ksplit > (g.K + kstep - 1) / kstep || g.part == nullptr) return cudaErrorInvalidValue;
            prm.part[q] = g.part;
            prm.part_cols[q] = mode == kGemmSwiGLU ? 2 * g.N : g.N;
        }
        prm.offsets[q] = g.offsets;
        prm.out[q] = g.out;
        prm.row_scale[q] = g.row_scale;
        prm.wscale1[q] = w8 ? g.wscale1 : nullptr;
        prm.wscale2[q] = w8 ? g.wscale2 : nullptr;
        prm.G[q] = g.G;
        prm.M[q] = g.M;
        prm.N[q] = g.N;
        prm.K[q] = g.K;
        prm.x_rows[q] = g.a_rows;
    }
    prm.nprob = nprob;
    prm.status = status;
    prm.wait_limit_ns = kWaitLimitNs;
    const char* stall = getenv("MOE_TEST_STALL_GEMM");
    if (stall && stall[0] == '1') {
        prm.stall_producer = 1;
        prm.wait_limit_ns = 20000000ull;
    }
    const int grid = num_sms > 0 ? num_sms : 148;
    if (mode == kGemmSwiGLU)
        return w8 ? launch_dec_nt<kGemmSwiGLU, true>(prm, nt, grid, s) : launch_dec_nt<kGemmSwiGLU, false>(prm, nt, grid, s);
    return w8 ? launch_dec_nt<kGemmScale, true>(prm, nt, grid, s) : launch_dec_nt<kGemmScale, false>(prm, nt, grid, s);
}

}  // namespace moe
