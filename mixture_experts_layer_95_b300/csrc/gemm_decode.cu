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
// D^T = W X^T.  A stage then holds a 256-row weight tile with 128-byte rows
// (32 KB: 64 bf16 or 128 FP8 codes of K per row) plus its NT token rows, so
// 4 to 6 stages -- 128 to 192 KB of weights -- stay in flight per SM.  The
// epilogue runs along the weight-row axis: the 32 lanes of a warp hold 32
// consecutive output columns, so every store of one token row is one
// contiguous segment.
//
// FP8 (E4M3) weights go to the tensor cores as they are (kind::f8f6f4, no
// widening pass); the token operand then has to be FP8 too, so every bf16
// token row arrives split as  x = s * (hi + lo)  with hi and lo E4M3 codes and
// s a power of two per row (split_e4m3 in fp8.cu), and each K step is two MMAs
// (hi, then lo) into the same accumulator.  The epilogue multiplies column j
// by s of its token row and row m by the weight row's scale.
//
// Roles: warp 0 TMA producer (weight tile + token rows, gathered with
// tile::gather4 when the rows come straight from the token matrix); warp 1
// TMEM allocation and the single MMA-issuing thread (two M=128 MMAs per K
// step, one per half of the weight tile; four with FP8 tokens); warps 2-5
// epilogue.  Split-K, per-row gates, FP8 per-channel scales and the bounded
// mbarrier waits are as in gemm_tc.cu.

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {
using namespace tc;

constexpr int WR = 256;                  // weight rows per tile (SwiGLU: 128 of W1 + 128 of W3)
// A stage carries KPS k-blocks of 64: 1 for bf16 weights; 2 for FP8, so that
// every weight row of a stage is 128 contiguous bytes (one 128-byte swizzle
// row, one full TMA row request) in both cases.
template <bool W8>
constexpr int kps() {
    return W8 ? 2 : 1;
}
constexpr int DEC_THREADS = 192;         // producer, MMA, 4 epilogue warps
constexpr int DEC_MAX_RING = 8;
constexpr int DEC_TMEM_COLS = 256;       // two accumulators of 2 x NT columns (NT <= 64)
constexpr int MAX_GROUPS = kMaxExperts;

struct DecParams {  // CUtensorMap members carry their own 64-byte alignment
    CUtensorMap tmX[2];   // token rows: a gather map (one-row box) or a tile map (NT-row box); FP8: hi codes
    CUtensorMap tmXlo[2]; // FP8: lo codes, same geometry
    CUtensorMap tmW1[2];  // weights: W1 (SwiGLU) or W2 (down)
    CUtensorMap tmW2[2];  // W3 (SwiGLU)
    const int32_t* offsets[2];
    void* out[2];
    int out_bf16[2];  // Scale mode without split-K: out holds bf16 rows
    const float* row_scale[2];
    const float* wscale1[2];
    const float* wscale2[2];
    const int32_t* x_gather[2];
    const float* x_scale[2];  // FP8: power-of-two scale of every token row (indexed like the token matrix)
    int G[2], M[2], N[2], K[2], x_rows[2], x_src_rows[2];
    float* part[2];
    int part_cols[2];
    int nprob, ksplit;
    // balanced split-K (ksplit 2, one problem): every CTA takes an equal,
    // contiguous share of all tiles' k-blocks, cut at tile boundaries; a
    // tile's part that starts at k-block 0 is slice 0, the rest slice 1 (a
    // tile one CTA covers whole writes zeros to slice 1)
    int balanced;
    // SwiGLU with split-K (non-null): one counter per output tile (zero
    // before the launch); the CTA that writes a tile's last K slice sums the
    // slices, applies SwiGLU and writes H itself, and resets the counter
    unsigned int* tile_sync;
    int* status;
    uint64_t wait_limit_ns;
    int stall_producer;
};

struct DecTail {
    uint64_t full[DEC_MAX_RING];
    uint64_t empty[DEC_MAX_RING];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint32_t tmem_base;
    int abort_flag;
    int fix_last;  // epilogue: this CTA wrote the current tile's last K slice
    int total[2];
    int gbase[2];
    int tile_start[MAX_GROUPS + 1];  // a group's rows come from the offsets (grp_rows)
};

constexpr int kSmemLimit = 232448;  // 227 KB opt-in per CTA

// A stage: the 256-row weight tile (128-byte rows), then the token tile(s):
// NT rows of 64 bf16, or NT rows of 128 hi codes and NT rows of 128 lo codes.
template <bool W8, int NT>
constexpr int dec_slot_bytes() {
    return WR * 128 + (W8 ? 2 : 1) * NT * 128;
}

constexpr int dec_fixed_bytes() { return 1024 + (int)sizeof(DecTail); }

template <bool W8, int NT>
constexpr int dec_stages() {
    return (kSmemLimit - dec_fixed_bytes()) / dec_slot_bytes<W8, NT>() > DEC_MAX_RING
               ? DEC_MAX_RING
               : (kSmemLimit - dec_fixed_bytes()) / dec_slot_bytes<W8, NT>();
}

template <bool W8, int NT>
constexpr size_t dec_smem_bytes() {
    return (size_t)dec_fixed_bytes() + (size_t)dec_stages<W8, NT>() * dec_slot_bytes<W8, NT>();
}

static_assert(dec_stages<false, 32>() >= 4 && dec_stages<false, 64>() >= 4, "bf16 decode ring too shallow");
static_assert(dec_stages<true, 32>() >= 4 && dec_stages<true, 64>() >= 4, "FP8 decode ring too shallow");
static_assert(dec_stages<true, 48>() >= 5 && dec_smem_bytes<true, 48>() <= kSmemLimit,
              "FP8 decode with 48 token rows: five stages");
static_assert(dec_smem_bytes<true, 32>() <= kSmemLimit && dec_smem_bytes<false, 64>() <= kSmemLimit &&
                  dec_smem_bytes<true, 64>() <= kSmemLimit && dec_smem_bytes<false, 32>() <= kSmemLimit,
              "decode GEMM exceeds shared memory");

struct DTile {
    int prob, g, m, n;
    int x_row0, rows_valid;
    int ks, kb0, kb1;  // K slice and its range of stages [kb0, kb1) (KPS k-blocks each)
    bool whole;        // balanced split-K: this CTA covers the whole K range (slice 1 gets zeros)
    int out_id;        // output tile (the tile-list entries of its K slices share it)
};

// output columns one tile covers: 128 (the W1/W3 pair) or 256 (W2)
template <int MODE>
__device__ __forceinline__ int dec_cols() {
    return MODE == kGemmSwiGLU ? WR / 2 : WR;
}

// Rows [lo, hi) of group g of problem q: its offsets, or all M rows; a range
// that does not fit the token matrix is empty (the tile scan records it).
__device__ __forceinline__ void grp_rows(const DecParams& p, int q, int g, int& lo, int& hi) {
    lo = 0;
    hi = p.M[q];
    if (p.offsets[q]) {
        lo = __ldg(p.offsets[q] + g);
        hi = __ldg(p.offsets[q] + g + 1);
    }
    if (lo < 0 || hi < lo || hi > p.x_rows[q]) lo = hi = 0;
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
    int row0, row1;
    grp_rows(p, t.prob, lo, row0, row1);
    const int rows = row1 - row0;
    const int mt = (rows + NT - 1) / NT;
    int r = local - ts[lo];
    const int units = p.balanced ? 1 : p.ksplit;  // tile-list entries per output tile
    t.ks = r % units;  // K slices of one output tile are adjacent, then token chunks
    r /= units;
    t.n = r / mt;
    t.m = r - t.n * mt;
    t.x_row0 = row0 + t.m * NT;
    t.rows_valid = min(NT, rows - t.m * NT);
    const int nk = (p.K[t.prob] + KPS * BK - 1) / (KPS * BK);
    t.kb0 = t.ks * nk / units;
    t.kb1 = (t.ks + 1) * nk / units;
    t.whole = p.balanced != 0;
    t.out_id = id / units;  // every group's and problem's entry count is a multiple of units
    return t;
}

// This CTA's work items, the same sequence for every role: tiles round-robin
// over the grid, or (balanced split-K, when every CTA's share is at least one
// whole tile) contiguous shares of the flattened (tile, k-block) space.
struct DecWork {
    long long pos, end;  // balanced: flat k-block positions; else pos = next tile id
    int nk;              // stages per tile (balanced)
    bool flat;
};

template <int KPS>
__device__ __forceinline__ DecWork dec_work_begin(const DecParams& p, int total_tiles) {
    DecWork w;
    w.nk = (p.K[0] + KPS * BK - 1) / (KPS * BK);
    const long long W = (long long)total_tiles * w.nk;
    w.flat = p.balanced && w.nk > 0 && W / gridDim.x >= w.nk;
    if (w.flat) {
        w.pos = (long long)blockIdx.x * W / gridDim.x;
        w.end = (long long)(blockIdx.x + 1) * W / gridDim.x;
    } else {
        w.pos = blockIdx.x;
        w.end = total_tiles;
    }
    return w;
}

template <int MODE, int NT, int KPS>
__device__ __forceinline__ bool dec_work_next(const DecTail& st, const DecParams& p, DecWork& w, DTile& t) {
    if (w.pos >= w.end) return false;
    if (!w.flat) {
        t = dec_tile<MODE, NT, KPS>(st, p, (int)w.pos);
        w.pos += gridDim.x;
        return true;
    }
    const int id = (int)(w.pos / w.nk);
    const int kb = (int)(w.pos - (long long)id * w.nk);
    const long long seg_end = min(w.end, (long long)(id + 1) * w.nk);
    t = dec_tile<MODE, NT, KPS>(st, p, id);
    t.kb0 = kb;
    t.kb1 = kb + (int)(seg_end - w.pos);
    t.ks = kb == 0 ? 0 : 1;
    t.whole = kb == 0 && t.kb1 == w.nk;
    w.pos = seg_end;
    return true;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

// FP8 tokens: the power-of-two scale of token column j of tile t (its row of
// the token matrix, through the gather list when there is one); 1 for bf16.
__device__ __forceinline__ float dec_xscale(const DecParams& p, const DTile& t, int j) {
    const float* xs = p.x_scale[t.prob];
    if (!xs) return 1.0f;
    const int r = t.x_row0 + j;
    const int32_t* gidx = p.x_gather[t.prob];
    int src = r;
    if (gidx) {
        src = __ldg(gidx + r);
        if (src < 0 || src >= p.x_src_rows[t.prob]) src = 0;  // recorded by the producer
    }
    return __ldg(xs + src);
}

// 32 accumulator columns from c0 on, or the last 16 when NT is not a
// multiple of 32 (NT = 48), so that a load never crosses into the next
// accumulator half.
template <int NT>
__device__ __forceinline__ void dec_tmem_ld(uint32_t taddr, int c0, uint32_t (&r)[32]) {
    if (NT % 32 != 0 && NT - c0 < 32) tmem_ld16(taddr, r);
    else tmem_ld32(taddr, r);
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
            dec_tmem_ld<NT>(tacc + c0, c0, g);
            dec_tmem_ld<NT>(tacc + NT + c0, c0, u);
            tmem_ld_wait();
            if (!live) continue;
            const int jn = min(32, t.rows_valid - c0);
            if (p.ksplit > 1) {
                const size_t pc = static_cast<size_t>(p.part_cols[t.prob]);
                float* base = p.part[t.prob] + (static_cast<size_t>(t.ks) * p.x_rows[t.prob] + t.x_row0 + c0) * pc;
                float* zero = t.whole && p.balanced
                                  ? p.part[t.prob] + ((size_t)p.x_rows[t.prob] + t.x_row0 + c0) * pc
                                  : nullptr;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < jn) {
                        const float xs = dec_xscale(p, t, c0 + j);
                        base[j * pc + f] = s1 * xs * __uint_as_float(g[j]);
                        base[j * pc + N + f] = s3 * xs * __uint_as_float(u[j]);
                        if (zero) {
                            zero[j * pc + f] = 0.f;
                            zero[j * pc + N + f] = 0.f;
                        }
                    }
            } else {
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[t.prob]) + (size_t)(t.x_row0 + c0) * N + f;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < jn) {
                        const float xs = dec_xscale(p, t, c0 + j);
                        out[(size_t)j * N] = __float2bfloat16_rn(
                            silu_mul(s1 * xs * __uint_as_float(g[j]), s3 * xs * __uint_as_float(u[j])));
                    }
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
                dec_tmem_ld<NT>(tacc + h * NT + c0, c0, v);
                tmem_ld_wait();
                if (!live) continue;
                const int jn = min(32, t.rows_valid - c0);
                const size_t row = (size_t)(t.x_row0 + c0);
                const float* rs = p.row_scale[t.prob] ? p.row_scale[t.prob] + row : nullptr;
                if (p.ksplit == 1 && p.out_bf16[t.prob]) {  // bf16 rows
                    __nv_bfloat16* db = static_cast<__nv_bfloat16*>(p.out[t.prob]) + row * N + o;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < jn)
                            db[(size_t)j * N] = __float2bfloat16_rn(
                                (rs ? __ldg(rs + j) : 1.0f) * dec_xscale(p, t, c0 + j) * ws * __uint_as_float(v[j]));
                    continue;
                }
                float* dst = p.ksplit > 1
                                 ? p.part[t.prob] + (static_cast<size_t>(t.ks) * p.x_rows[t.prob] + row) * N + o
                                 : static_cast<float*>(p.out[t.prob]) + row * N + o;
                float* zero = p.ksplit > 1 && t.whole && p.balanced
                                  ? p.part[t.prob] + ((size_t)p.x_rows[t.prob] + row) * N + o
                                  : nullptr;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < jn) {
                        dst[(size_t)j * N] =
                            (rs ? __ldg(rs + j) : 1.0f) * dec_xscale(p, t, c0 + j) * ws * __uint_as_float(v[j]);
                        if (zero) zero[(size_t)j * N] = 0.f;
                    }
            }
        }
    }
}

// Split-K SwiGLU finished by the CTA that wrote an output tile's last K
// slice: for this thread's hidden channel f, every token row of the tile sums
// its K slices in slice order (the other CTAs' partials read through L2) and
// becomes silu(g) * u in bf16 -- the arithmetic of swiglu_finalize_kernel, in
// the same order, so H is bit-identical to the separate pass it replaces.
template <int NT>
__device__ __forceinline__ void dec_swiglu_fixup(const DecParams& p, const DTile& t, int wrow) {
    const int N = p.N[t.prob];
    const int f = t.n * (WR / 2) + wrow;
    if (f >= N) return;
    const size_t pc = static_cast<size_t>(p.part_cols[t.prob]);
    const size_t stride = static_cast<size_t>(p.x_rows[t.prob]) * pc;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[t.prob]);
    for (int j = 0; j < t.rows_valid; ++j) {
        const size_t row = static_cast<size_t>(t.x_row0 + j);
        const float* gp = p.part[t.prob] + row * pc + f;
        float g = __ldcg(gp), u = __ldcg(gp + N);
        for (int sl = 1; sl < p.ksplit; ++sl) {
            g += __ldcg(gp + sl * stride);
            u += __ldcg(gp + sl * stride + N);
        }
        out[row * N + f] = __float2bfloat16_rn(g / (1.0f + __expf(-g)) * u);
    }
}

template <int MODE, bool W8, int NT>
__global__ void __launch_bounds__(DEC_THREADS, 1) grouped_gemm_decode_kernel(const __grid_constant__ DecParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int NST = dec_stages<W8, NT>();
    constexpr int SLOT = dec_slot_bytes<W8, NT>();
    constexpr int KPS = kps<W8>();
    constexpr int WBYTES = WR * 128;  // weight bytes at the start of a stage
    constexpr int XBYTES = NT * 128;  // one token tile: NT rows of 128 bytes
    static_assert(MODE == kGemmSwiGLU || MODE == kGemmScale, "decode GEMM: SwiGLU and Scale modes");
    DecTail& st = *reinterpret_cast<DecTail*>(smem + (size_t)NST * SLOT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &st.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&st.full[s], 1);
            mbar_init(&st.empty[s], 1);
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
            if (W8) prefetch_tmap(&p.tmXlo[q]);
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
                        int lo, hi;
                        grp_rows(p, q, g, lo, hi);
                        if (p.offsets[q]) {  // report a range grp_rows emptied
                            const int a = p.offsets[q][g], b = p.offsets[q][g + 1];
                            if (a < 0 || b < a || b > p.x_rows[q]) record_status(p.status, kStatusBounds);
                        }
                        tiles = ((hi - lo + NT - 1) / NT) * ncb * (p.balanced ? 1 : p.ksplit);
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
        // ---------------- TMA producer: weight tile + token rows per stage ----------------
        int s = 0;
        uint32_t ph = 0;
        uint32_t issued_parity[NST];
        bool used[NST];
        for (int i = 0; i < NST; ++i) used[i] = false;
        bool dead = p.stall_producer != 0;
        DecWork work = dec_work_begin<KPS>(p, total_tiles);
        DTile t;
        while (!dead && dec_work_next<MODE, NT, KPS>(st, p, work, t)) {
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
            // token bytes of one tile: gathered rows come in groups of four
            const uint32_t x_bytes = gidx ? (uint32_t)((t.rows_valid + 3) / 4) * 4 * 128 : (uint32_t)XBYTES;
            for (int kb = t.kb0; kb < t.kb1; ++kb) {
                if (!mbar_wait(&st.empty[s], ph ^ 1u, abort_flag, p.status, p.wait_limit_ns)) {
                    dead = true;
                    break;
                }
                uint8_t* sw = smem + (size_t)s * SLOT;
                // KPS * 64 elements of K: 64 bf16 or 128 FP8 codes, 128 bytes per row either way
                const int kc = kb * KPS * BK;
                if (lane == 0) {
                    mbar_expect_tx(&st.full[s], WBYTES + (W8 ? 2u : 1u) * x_bytes);
                    if (MODE == kGemmSwiGLU) {
                        tma_load_2d(sw, &p.tmW1[t.prob], kc, w_row0, &st.full[s]);
                        tma_load_2d(sw + WBYTES / 2, &p.tmW2[t.prob], kc, w_row0, &st.full[s]);
                    } else {
                        tma_load_2d(sw, &p.tmW1[t.prob], kc, w_row0, &st.full[s]);
                    }
                    if (!gidx) {
                        tma_load_2d(sw + WBYTES, &p.tmX[t.prob], kc, t.x_row0, &st.full[s]);
                        if (W8) tma_load_2d(sw + WBYTES + XBYTES, &p.tmXlo[t.prob], kc, t.x_row0, &st.full[s]);
                    }
                }
                if (gidx && lane * 4 < t.rows_valid) {
                    tma_gather4(sw + WBYTES + lane * 4 * 128, &p.tmX[t.prob], kc, rows4[0], rows4[1], rows4[2],
                                rows4[3], &st.full[s]);
                    if (W8)
                        tma_gather4(sw + WBYTES + XBYTES + lane * 4 * 128, &p.tmXlo[t.prob], kc, rows4[0], rows4[1],
                                    rows4[2], rows4[3], &st.full[s]);
                }
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
            constexpr uint32_t idesc = W8 ? idesc_e4m3_f32(128, NT) : idesc_bf16_f32(128, NT);
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool dead = false;
            DecWork work = dec_work_begin<KPS>(p, total_tiles);
            DTile t;
            for (; !dead && dec_work_next<MODE, NT, KPS>(st, p, work, t); ++it) {
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
                    tc_fence_after();
                    const uint32_t sw = smem_u32(smem + (size_t)s * SLOT);
                    const uint32_t sx = sw + WBYTES;
                    // four 32-byte K steps per 128-byte row: 16 bf16 or 32 FP8 codes each
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t accf = (kb != t.kb0 || kk != 0) ? 1u : 0u;
                        const uint64_t a0 = sdesc_k_sw128(sw + kk * 32);
                        const uint64_t a1 = sdesc_k_sw128(sw + 128 * 128 + kk * 32);
                        const uint64_t xh = sdesc_k_sw128(sx + kk * 32);
                        if constexpr (W8) {  // tokens as hi + lo codes: two MMAs per weight half
                            const uint64_t xl = sdesc_k_sw128(sx + XBYTES + kk * 32);
                            umma_e4m3(dtm, a0, xh, idesc, accf);
                            umma_e4m3(dtm, a0, xl, idesc, 1u);
                            umma_e4m3(dtm + NT, a1, xh, idesc, accf);
                            umma_e4m3(dtm + NT, a1, xl, idesc, 1u);
                        } else {
                            umma_bf16(dtm, a0, xh, idesc, accf);
                            umma_bf16(dtm + NT, a1, xh, idesc, accf);
                        }
                    }
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
    } else {
        // ---------------- epilogue (warps 2..5): one weight row per thread ----------------
        const int quarter = warp & 3;
        const int wrow = quarter * 32 + lane;
        int it = 0;
        DecWork work = dec_work_begin<KPS>(p, total_tiles);
        DTile t;
        for (; dec_work_next<MODE, NT, KPS>(st, p, work, t); ++it) {
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
            if (MODE == kGemmSwiGLU && p.tile_sync) {
                // count this slice in once all four epilogue warps have written it
                __threadfence();
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (warp == 2 && lane == 0) {
                    const unsigned int mine = (p.balanced && t.whole) ? 2u : 1u;  // slices this CTA wrote
                    int last = 1;
                    if (mine < (unsigned int)p.ksplit) {
                        const unsigned int before = atomicAdd(p.tile_sync + t.out_id, mine);
                        last = before + mine == (unsigned int)p.ksplit;
                        if (last) p.tile_sync[t.out_id] = 0u;  // every slice is in: ready for the next launch
                    }
                    st.fix_last = last;
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (st.fix_last) {
                    __threadfence();
                    dec_swiglu_fixup<NT>(p, t, wrow);
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
    launch_pdl(grouped_gemm_decode_kernel<MODE, W8, NT>, dim3(grid), dim3(DEC_THREADS),
               dec_smem_bytes<W8, NT>(), s, prm);
    return cudaGetLastError();
}

template <int MODE, bool W8>
cudaError_t launch_dec_nt(const DecParams& prm, int nt, int grid, cudaStream_t s) {
    if (nt == 48) return W8 ? launch_dec<MODE, true, 48>(prm, grid, s) : cudaErrorInvalidValue;
    return nt == 32 ? launch_dec<MODE, W8, 32>(prm, grid, s) : launch_dec<MODE, W8, 64>(prm, grid, s);
}

}  // namespace

cudaError_t launch_gemm_decode(int mode, const GemmProblem* probs, int nprob, int* status, int num_sms,
                               cudaStream_t s, int ksplit, bool w8, int nt, bool balanced, unsigned int* tile_sync) {
    if (balanced && (ksplit != 2 || nprob != 1)) return cudaErrorInvalidValue;
    if (tile_sync && (mode != kGemmSwiGLU || ksplit < 2)) return cudaErrorInvalidValue;
    if (nprob < 1 || nprob > 2 || ksplit < 1 || (nt != 32 && nt != 64 && !(nt == 48 && w8)))
        return cudaErrorInvalidValue;
    if (mode != kGemmSwiGLU && mode != kGemmScale) return cudaErrorInvalidValue;
    DecParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.ksplit = ksplit;
    const int w_box = mode == kGemmSwiGLU ? WR / 2 : WR;
    if (probs[0].G + (nprob > 1 ? probs[1].G : 0) > MAX_GROUPS + 1) return cudaErrorInvalidValue;
    for (int q = 0; q < nprob; ++q) {
        const GemmProblem& g = probs[q];
        if (g.G < 1 || g.G > MAX_GROUPS || g.out2 || g.b_mn) return cudaErrorInvalidValue;
        // FP8: A holds the hi codes of the tokens, A2 the lo codes, a_scale the row scales
        if (w8 && (g.K % 16 != 0 || !g.wscale1 || (mode == kGemmSwiGLU && !g.wscale2) || !g.A2 || !g.a_scale))
            return cudaErrorInvalidValue;
        if (!w8 && (g.A2 || g.a_scale)) return cudaErrorInvalidValue;
        const int x_src = g.a_gather ? g.a_src_rows : g.a_rows;
        const int x_box = g.a_gather ? 1 : nt;  // gather maps: one-row box
        if (w8) {  // FP8 stages hold 128 codes (two k-blocks) of every weight and token row
            if (!make_tmap_u8(&prm.tmX[q], g.A, x_src, g.K, x_box, 2 * BK, true) ||
                !make_tmap_u8(&prm.tmXlo[q], g.A2, x_src, g.K, x_box, 2 * BK, true) ||
                !make_tmap_u8(&prm.tmW1[q], g.B1, g.G * g.N, g.K, w_box, 2 * BK, true) ||
                (mode == kGemmSwiGLU && !make_tmap_u8(&prm.tmW2[q], g.B2, g.G * g.N, g.K, w_box, 2 * BK, true)))
                return cudaErrorInvalidValue;
            prm.x_scale[q] = g.a_scale;
        } else {
            if (!make_tmap(&prm.tmX[q], g.A, x_src, g.K, x_box) ||
                !make_tmap(&prm.tmW1[q], g.B1, g.G * g.N, g.K, w_box) ||
                (mode == kGemmSwiGLU && !make_tmap(&prm.tmW2[q], g.B2, g.G * g.N, g.K, w_box)))
                return cudaErrorInvalidValue;
        }
        if (g.a_gather) {
            prm.x_gather[q] = g.a_gather;
            prm.x_src_rows[q] = g.a_src_rows;
        }
        if (ksplit > 1) {
            const int kstep = (w8 ? 2 : 1) * BK;
            if (ksplit > (g.K + kstep - 1) / kstep || g.part == nullptr) return cudaErrorInvalidValue;
            prm.part[q] = g.part;
            prm.part_cols[q] = mode == kGemmSwiGLU ? 2 * g.N : g.N;
        }
        if (g.out_bf16 && mode != kGemmScale) return cudaErrorInvalidValue;
        prm.offsets[q] = g.offsets;
        prm.out[q] = g.out;
        prm.out_bf16[q] = g.out_bf16;
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
    prm.balanced = balanced ? 1 : 0;
    prm.tile_sync = tile_sync;
    prm.status = status;
    prm.wait_limit_ns = kWaitLimitNs;
    if (test_stall_gemm()) {
        prm.stall_producer = 1;
        prm.wait_limit_ns = kStallWaitLimitNs;
    }
    const int grid = num_sms > 0 ? num_sms : 148;
    if (mode == kGemmSwiGLU)
        return w8 ? launch_dec_nt<kGemmSwiGLU, true>(prm, nt, grid, s) : launch_dec_nt<kGemmSwiGLU, false>(prm, nt, grid, s);
    return w8 ? launch_dec_nt<kGemmScale, true>(prm, nt, grid, s) : launch_dec_nt<kGemmScale, false>(prm, nt, grid, s);
}

}  // namespace moe
