// gemm_tc.cu -- grouped expert GEMMs on the 5th-generation tensor cores.
//
// "Mixture of experts (MoE)" handbook, "Implementation: token by token vs.
// grouped by expert": each expert does one matrix multiplication over all the
// tokens assigned to it (its contiguous segment after grouping), and "one
// grouped GEMM computes all the experts at once".  The expert itself is the
// handbook's SwiGLU Expert (down(silu(gate(x)) * up(x))), so one layer call
// runs two grouped GEMMs:
//   up:   H[r, :]  = silu(X[r] W1_g^T) * (X[r] W3_g^T)     (bf16 out)
//   down: Y[r, :]  = gate[r] * (H[r] W2_g^T)                (fp32 out)
// for every row r of group g's segment, plus the same for the shared expert
// as a second problem in the same launch.  The router's logits (x W_g^T,
// fp32 out) reuse the kernel with a single group.
//
// Design (sm_103a):
//  * persistent: one CTA per SM walks a device-side tile list derived from the
//    group offsets (no host sync); tiles are 128 rows x 256 accumulator
//    columns; consecutive tiles share a weight tile (row blocks vary fastest)
//    so that each weight tile is fetched from HBM once and re-read from L2.
//  * warp 0: TMA producer (cp.async.bulk.tensor, 128-byte swizzle, 4-stage
//    mbarrier ring; rows past a segment's end are loaded but never stored,
//    rows past the tensor are zero-filled by the TMA unit).  For decode-sized
//    batches the up GEMM of the fused layer gathers its A rows straight from
//    the token matrix with tile::gather4 (4 rows per load, indices from the
//    permutation, only the tile's valid rows), so no permuted copy of x is
//    written; large batches load A as plain tiles of that copy, because 32
//    gather4 loads per 16 KB stage cannot keep up with the tensor cores.
//  * warp 1: allocates 512 TMEM columns (two 128x256 fp32 accumulators) and
//    one lane issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, M=128,
//    N=256, K=16 per instruction); tcgen05.commit frees smem stages and
//    hands finished accumulators to the epilogue.
//  * warps 2-5: epilogue; tcgen05.ld 32 columns at a time, fused SwiGLU /
//    gate scaling, 16-byte stores.  The two accumulators let the epilogue of
//    tile i overlap the main loop of tile i+1.
//  * every mbarrier wait is bounded (%globaltimer); on expiry the CTA records
//    MOE_ERR_TIMEOUT in the status word, stops issuing work, waits (bounded)
//    for its copies in flight, frees its TMEM and returns.
#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {
using namespace tc;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int STAGES = 4;  // ring depth; 3 for the split-A down GEMM (64 KB stages)
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;

// Per-mode stage layout: [A | (A_lo) | B].  The split mode multiplies two A
// operands (the hi and lo bf16 halves of H) by the same B tile.
template <int MODE>
struct StageCfg {
    static constexpr bool kSplit = MODE == kGemmScaleSplit;
    static constexpr int kStages = kSplit ? 3 : STAGES;
    static constexpr int kBOff = kSplit ? 2 * A_BYTES : A_BYTES;
    static constexpr int kBytes = kBOff + B_BYTES;
};
constexpr int NUM_THREADS = 192;
// FP8-weight variant: 4 more warps (6..9) widen the raw one-byte B tiles
constexpr int W8_THREADS = NUM_THREADS + 128;
constexpr int F8_BYTES = BN * BK;   // 256 weight rows x 64 one-byte elements
constexpr int W8_RAW = 4;           // TMA stages in flight: bf16 A tile + one-byte B tile
constexpr int W8_RAW_BYTES = A_BYTES + F8_BYTES;
constexpr int W8_WIDE = 2;          // widened bf16 B tiles feeding the MMA
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_GROUPS = kMaxExperts;

struct TcParams {  // CUtensorMap members carry their own 64-byte alignment
    CUtensorMap tmA[2];
    CUtensorMap tmA2[2];  // split mode: the lo half of A
    CUtensorMap tmB1[2];
    CUtensorMap tmB2[2];
    const int32_t* offsets[2];
    void* out[2];
    int out_bf16[2];  // fp32-accumulator modes: out holds bf16 rows
    void* out2[2];  // SwiGLU: when non-null, the lo half of H (H - bf16(H)) goes here
    const float* row_scale[2];
    int G[2], M[2], N[2], K[2], a_rows[2];
    const int32_t* a_gather[2];  // non-null: A row r is row a_gather[r] of tmA's tensor (gather4 loads)
    int a_src_rows[2];           // rows of the tensor tmA describes when gathering
    int nprob;
    int ksplit;                // K slices per tile (1: no split)
    float* part[2];            // ksplit > 1: fp32 partials [ksplit][a_rows][part_cols]
    int part_cols[2];          // 2N for SwiGLU (gate half, then up half), N otherwise
    const float* wscale1[2];   // FP8 weights: per weight-row scale of B1 / B2 (null: bf16 weights)
    const float* wscale2[2];
    // K-grouped problem (non-null): every group g multiplies the same A rows
    // [0, M) by the same B rows [0, N) over its own K window [kbase[g],
    // kbase[g] + klen[g]) (kbase a multiple of 64; the operands hold zeros up
    // to the next multiple of 64) and writes output rows g*M .. g*M + M - 1
    const int32_t* kbase[2];
    const int32_t* klen[2];
    // MN-major B (Plain and Scale modes): tmB1 / tmB2 are 3-D maps {N, K, G}
    // of matrices stored [G][K][N] (B^T per group), loaded as 64x64 boxes.
    // kpart[q] > 0 splits K into two parts of kpart[q] each, every part padded
    // to whole k-blocks: part 0 reads A part 0 and tmB1, part 1 A part 1 and
    // tmB2, where tmA is then a 3-D map {kpart, 2, rows} of A = [rows][2 kpart].
    int b_mn;
    int kpart[2];
    // SwiGLU mode: when non-null, the fp32 G and U ([rows][N] each) go here too
    float* out_g[2];
    float* out_u[2];
    // kGemmSwigluBwd epilogue operands (GemmProblem::bwd_*); on CTA pairs G and
    // U also come in through tmG / tmU (fp32 [rows][N], 32 x 32 boxes, 128-byte swizzle)
    CUtensorMap tmG[2];
    CUtensorMap tmU[2];
    // ... and dG, dU, H go out through tmdG / tmdU / tmH (bf16 rows of bwd_dGU and
    // bwd_Hb, 32 x 32 boxes, 64-byte swizzle)
    CUtensorMap tmdG[2];
    CUtensorMap tmdU[2];
    CUtensorMap tmH[2];
    // columns of the MMA and of the B tile in Plain mode: BN, or 64 for a
    // product with N <= 64 (the router's logits GEMM), whose B box is then
    // 64 rows high
    int mma_n;
    const float* bwd_G[2];
    const float* bwd_U[2];
    __nv_bfloat16* bwd_dGU[2];
    __nv_bfloat16* bwd_Hb[2];
    float* bwd_dgp_part[2];
    int bwd_dgp_ld[2];
    int* status;
    uint64_t wait_limit_ns;  // bound on every mbarrier wait
    int stall_producer;      // test switch: issue no loads, so the consumers' bounded waits run out
    // CTA pairs: a group's last tile, when it holds at most 128 rows, is an
    // M = 128 MMA (64 rows per CTA) instead of M = 256.  One SM: a tile of at
    // most 64 rows is an M = 64 MMA instead of M = 128.
    int pair_half;
    int m64;
};

constexpr int kMaxRing = 6;  // deepest ring of any kernel here (the 2-SM kernel)

template <int NG>
struct SmemTailT {
    uint64_t full[kMaxRing];
    uint64_t empty[kMaxRing];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t wfull[W8_WIDE];   // FP8 variant: widened B tile ready for the MMA
    uint64_t wempty[W8_WIDE];  // FP8 variant: the MMA is done with a widened B tile
    uint32_t tmem_base;
    int abort_flag;
    int total[2];
    int gbase[2];  // first entry of each problem's groups in the arrays below
    // per group (both problems back to back; the launcher keeps G0 + G1 <= NG)
    int tile_start[NG];
    int row0[NG];
    int rows[NG];
    // CTA-pair SwiGLU backward: each epilogue warp's two G/U staging slots
    uint64_t gu_full[4][2];
};
using SmemTailCore = SmemTailT<MAX_GROUPS + 1>;
struct SmemTail : SmemTailCore {
    // epilogue staging: each epilogue warp passes 32 rows x 32 fp32 columns
    // through its block so that its global stores cover whole row segments
    alignas(16) float stage[4][32][33];
};

template <int MODE, bool W8>
constexpr int ring_stages() {
    return W8 ? W8_RAW : StageCfg<MODE>::kStages;
}

// bytes of one TMA ring stage
template <int MODE, bool W8>
constexpr int slot_bytes() {
    return W8 ? W8_RAW_BYTES : StageCfg<MODE>::kBytes;
}

// offset of the B tile inside a ring stage
template <int MODE, bool W8>
constexpr int slot_b_off() {
    return W8 ? A_BYTES : StageCfg<MODE>::kBOff;
}

template <int MODE, bool W8>
constexpr size_t smem_bytes() {
    return 1024 /*align slack*/ + (size_t)ring_stages<MODE, W8>() * slot_bytes<MODE, W8>() +
           (W8 ? (size_t)W8_WIDE * B_BYTES : 0) + sizeof(SmemTail);
}

// ------------------------------------------------------------- tile schedule

struct Tile {
    int prob, g, m, n;
    int a_row0, rows_valid;
    int ks, kb0, kb1;  // K slice and its k-block range [kb0, kb1)
    int out_row0;      // first output row (a_row0 except for K-grouped problems)
    int k_off;         // K coordinate of k-block 0 (K-grouped problems: the group's window)
    int half;          // CTA-pair tail tile of M = 128 (64 rows per CTA) instead of 256
};

template <int MODE>
__device__ __forceinline__ int out_cols_per_tile() {
    return MODE == kGemmSwiGLU ? BN / 2 : BN;
}

// 64-deep k-blocks of one tile's K range (two padded parts when kpart is set)
__device__ __forceinline__ int k_blocks(const TcParams& p, int prob) {
    return p.kpart[prob] ? 2 * ((p.kpart[prob] + BK - 1) / BK) : (p.K[prob] + BK - 1) / BK;
}

// MN-major B: loads k-block kb of a tile -- A (BM rows, plain or part-split)
// and nblk 64-column blocks of B^T starting at column n0 of group g -- onto
// `bar`.  load3 / load2 issue one 3-D / 2-D TMA copy.
template <typename Load3, typename Load2>
__device__ __forceinline__ void load_kblock_bmn(const TcParams& p, int prob, int kb, int a_row0, int n0, int g,
                                                int nblk, uint8_t* sa, uint8_t* sb, Load3 load3, Load2 load2) {
    const int nkp = p.kpart[prob] ? (p.kpart[prob] + BK - 1) / BK : 1 << 30;
    const int part = kb >= nkp ? 1 : 0;
    const int k0 = (kb - part * nkp) * BK;
    if (p.kpart[prob]) load3(sa, &p.tmA[prob], k0, part, a_row0);
    else load2(sa, &p.tmA[prob], k0, a_row0);
    const CUtensorMap* tb = part ? &p.tmB2[prob] : &p.tmB1[prob];
    for (int j = 0; j < nblk; ++j) load3(sb + j * (BK * BK * 2), tb, n0 + j * BK, k0, g);
}

template <int MODE>
__device__ __forceinline__ Tile decode_tile(const SmemTailCore& st, const TcParams& p, int id) {
    Tile t;
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
    const int mt = (rows + BM - 1) / BM;
    int r = local - ts[lo];
    t.ks = r % p.ksplit;  // K slices of one output tile are adjacent in the list
    r /= p.ksplit;
    t.n = r / mt;
    t.m = r - t.n * mt;
    t.a_row0 = st.row0[gb + lo] + t.m * BM;
    t.rows_valid = min(BM, rows - t.m * BM);
    t.out_row0 = t.a_row0;
    t.k_off = 0;
    t.half = (p.m64 && t.rows_valid <= BM / 2) ? 1 : 0;
    int nk = k_blocks(p, t.prob);
    if (p.kbase[t.prob]) {  // K-grouped: shared A rows, the group's own K window
        t.out_row0 = t.g * p.M[t.prob] + t.m * BM;
        t.k_off = __ldg(p.kbase[t.prob] + t.g);
        nk = (__ldg(p.klen[t.prob] + t.g) + BK - 1) / BK;
    }
    t.kb0 = t.ks * nk / p.ksplit;
    t.kb1 = (t.ks + 1) * nk / p.ksplit;
    return t;
}

// --------------------------------------------------------------- epilogues

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

// Split-K epilogue: the raw fp32 accumulator of this K slice goes to the
// partial buffer (scaled by the row's gate in the scale modes); a later pass
// sums the slices in slice order.  For SwiGLU the gate half lands in columns
// [0, N) and the up half in [N, 2N).
template <int MODE>
__device__ __forceinline__ void epilogue_partial(const TcParams& p, const Tile& t, uint32_t tacc, int row_in_tile,
                                                 int ncols = BN) {
    const int N = p.N[t.prob];
    const bool valid = row_in_tile < t.rows_valid;
    const size_t grow = static_cast<size_t>(t.out_row0 + row_in_tile);
    const size_t pc = static_cast<size_t>(p.part_cols[t.prob]);
    float* base = p.part[t.prob] + (static_cast<size_t>(t.ks) * p.a_rows[t.prob] + grow) * pc;
    float scale = 1.0f;
    if ((MODE == kGemmScale || MODE == kGemmScaleSplit) && valid && p.row_scale[t.prob] != nullptr)
        scale = __ldg(p.row_scale[t.prob] + grow);
#pragma unroll 1
    for (int c0 = 0; c0 < ncols; c0 += 32) {
        uint32_t v[32];
        __syncwarp();
        tmem_ld32(tacc + c0, v);
        tmem_ld_wait();
        int col;
        if (MODE == kGemmSwiGLU)
            col = (c0 < BN / 2) ? t.n * (BN / 2) + c0 : N + t.n * (BN / 2) + (c0 - BN / 2);
        else
            col = t.n * BN + c0;
        const int lim = (MODE == kGemmSwiGLU && c0 >= BN / 2) ? 2 * N : N;
        if (!valid || col >= lim) continue;
        {
            const bool up_half = MODE == kGemmSwiGLU && c0 >= BN / 2;
            const float* ws = up_half ? p.wscale2[t.prob] : p.wscale1[t.prob];
            const int wc = up_half ? col - N : col;  // weight row within the group
            if (ws) apply_wscale32(v, ws, static_cast<size_t>(t.g) * N + wc, N - wc);
        }
        float* dst = base + col;
        if (col + 32 <= lim) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                reinterpret_cast<float4*>(dst)[q] =
                    make_float4(scale * __uint_as_float(v[4 * q]), scale * __uint_as_float(v[4 * q + 1]),
                                scale * __uint_as_float(v[4 * q + 2]), scale * __uint_as_float(v[4 * q + 3]));
        } else {
            for (int i = 0; i < 32 && col + i < lim; ++i) dst[i] = scale * __uint_as_float(v[i]);
        }
    }
}

// SwiGLU backward of one row's 32 columns: with a = G, b = U, s = sigmoid(a)
// and dd = D (the upstream gradient of H), H = a s b, dG = g dd b s (1 + a (1 - s))
// and dU = g dd a s, packed as bf16 pairs (8 columns per uint4); the gate
// gradient's partial sum gains dd H over the first nc (<= 32) columns.
__device__ __forceinline__ void swiglu_bwd_pack(const float (&ga)[32], const float (&ub)[32], const uint32_t (&v)[32],
                                                int nc, float g, uint4 (&pg)[4], uint4 (&pu)[4], uint4 (&ph)[4],
                                                float& part) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float dG[8], dU[8], hh[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float a = ga[8 * q + i], b = ub[8 * q + i];
            const float dd = __uint_as_float(v[8 * q + i]);
            const float sg = __fdividef(1.0f, 1.0f + __expf(-a));  // (0 once exp(-a) passes 2^126)
            hh[i] = a * sg * b;
            if (8 * q + i < nc) part += dd * hh[i];
            const float dh = g * dd;
            dG[i] = dh * b * sg * (1.0f + a * (1.0f - sg));
            dU[i] = dh * a * sg;
        }
        uint32_t* wg = reinterpret_cast<uint32_t*>(&pg[q]);
        uint32_t* wu = reinterpret_cast<uint32_t*>(&pu[q]);
        uint32_t* wh = reinterpret_cast<uint32_t*>(&ph[q]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 x = __floats2bfloat162_rn(dG[2 * i], dG[2 * i + 1]);
            __nv_bfloat162 y = __floats2bfloat162_rn(dU[2 * i], dU[2 * i + 1]);
            __nv_bfloat162 z = __floats2bfloat162_rn(hh[2 * i], hh[2 * i + 1]);
            wg[i] = *reinterpret_cast<uint32_t*>(&x);
            wu[i] = *reinterpret_cast<uint32_t*>(&y);
            wh[i] = *reinterpret_cast<uint32_t*>(&z);
        }
    }
}

// The first nc (<= 32) of 32 packed bf16 values to out (16-byte aligned when nc == 32).
__device__ __forceinline__ void store_bf16_row(const uint4 (&w)[4], int nc, __nv_bfloat16* out) {
    if (nc == 32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) reinterpret_cast<uint4*>(out)[q] = w[q];
        return;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        if (i >= nc) break;
        const uint32_t word = (&w[i >> 3].x)[(i & 7) >> 1];
        out[i] = __ushort_as_bfloat16(static_cast<unsigned short>((i & 1) ? word >> 16 : word & 0xffffu));
    }
}

// The thread's accumulator row covers output columns [col_lo, col_lo + ncols)
// of the tile, at TMEM columns [0, ncols): the whole 256-column tile, or one
// half of it in a CTA-pair M = 128 tile, whose rows hold the first half of
// the columns in TMEM lanes 0-63 and the second half in lanes 64-127.
// ilv (CTA pairs, SwiGLU): the tile's columns are [W1 | W3] per 64 features,
// i.e. G of features 0-63, U of 0-63, G of 64-127, U of 64-127, so that
// either column half holds G and U of the same features.
// warp_row0 >= 0: the warp's rows are warp_row0 .. warp_row0 + warp_rows - 1,
// held by its lanes 0 .. warp_rows - 1 (an M = 64 tile keeps 16 rows in each
// 32-lane quarter of TMEM); otherwise the warp holds 32 consecutive rows.
// The warp's 32 rows x 32 fp32 columns (x: this thread's row, as bits) to
// dst + r * ld for the rows r < nvalid that exist and the columns c < ncv,
// through the warp's 32 x 32 shared block: row r's 16-byte chunk j sits at
// float r * 32 + ((j ^ (r & 7)) << 2), so that the row-wise 16-byte writes
// and the 16-byte reads of 8 lanes per row hit distinct banks and every store
// instruction covers 4 whole row segments.
__device__ __forceinline__ void stage_rows_f32(float* sb, const uint32_t (&x)[32], float* dst, size_t ld, int nvalid,
                                               int ncv) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(sb + lane * 32 + ((j ^ (lane & 7)) << 2)) =
            make_float4(__uint_as_float(x[4 * j]), __uint_as_float(x[4 * j + 1]), __uint_as_float(x[4 * j + 2]),
                        __uint_as_float(x[4 * j + 3]));
    __syncwarp();
    if (nvalid == 32 && ncv >= 32 && (ld & 3) == 0) {
        const int rq = lane >> 3, jj = lane & 7;
        float4 q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + rq;
            q[i] = *reinterpret_cast<const float4*>(sb + rr * 32 + ((jj ^ (rr & 7)) << 2));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) *reinterpret_cast<float4*>(dst + (size_t)(4 * i + rq) * ld + 4 * jj) = q[i];
    } else if (lane < ncv) {
        for (int r = 0; r < nvalid; ++r)
            dst[(size_t)r * ld + lane] = sb[r * 32 + (((lane >> 2) ^ (r & 7)) << 2) + (lane & 3)];
    }
    __syncwarp();  // the block is read before it is written again
}

// W8: the FP8-weight kernel, which never keeps G and U (no out_g / out_u)
template <int MODE, bool W8 = false>
__device__ __forceinline__ void epilogue_tile(const TcParams& p, const Tile& t, uint32_t tacc, int row_in_tile,
                                              float (*stage)[33], int col_lo = 0, int ncols = BN, bool ilv = false,
                                              int warp_row0 = -1, int warp_rows = 32) {
    if (MODE == kGemmPlain && p.mma_n < ncols) ncols = p.mma_n;  // (columns past mma_n hold nothing)
    if (p.ksplit > 1) {
        epilogue_partial<MODE>(p, t, tacc, row_in_tile, ncols);
        return;
    }
    const int N = p.N[t.prob];
    const bool valid = row_in_tile < t.rows_valid;
    const size_t grow = static_cast<size_t>(t.out_row0 + row_in_tile);
    if (MODE == kGemmSwiGLU) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[t.prob]);
        __nv_bfloat16* out_lo = static_cast<__nv_bfloat16*>(p.out2[t.prob]);
        const int nchunks = ilv ? ncols / 64 : BN / 2 / 32;
        const int wrow0 = warp_row0 >= 0 ? warp_row0 : row_in_tile - (int)(threadIdx.x & 31);  // first row of this warp
        const int nvalid = min(warp_rows, t.rows_valid - wrow0);                                 // its rows that exist
#pragma unroll 1
        for (int ch = 0; ch < nchunks; ++ch) {
            int gcol, ucol, col;  // TMEM columns of G and U, first output feature
            if (ilv) {
                const int b = (ch >> 1) * 128, c0 = (ch & 1) * 32;
                gcol = b + c0;
                ucol = b + 64 + c0;
                col = t.n * (BN / 2) + ((col_lo + b) >> 1) + c0;
            } else {
                gcol = ch * 32;
                ucol = BN / 2 + ch * 32;
                col = t.n * (BN / 2) + ch * 32;
            }
            uint32_t g[32], u[32];
            __syncwarp();  // tcgen05.ld is warp-aligned: reconverge after the per-lane stores
            tmem_ld32(tacc + gcol, g);
            tmem_ld32(tacc + ucol, u);
            tmem_ld_wait();
            if (col >= N) continue;  // (uniform across the warp)
            if (p.wscale1[t.prob]) {  // FP8 weights: per-channel scales of W1 and W3
                const size_t wr = static_cast<size_t>(t.g) * N + col;
                apply_wscale32(g, p.wscale1[t.prob], wr, N - col);
                apply_wscale32(u, p.wscale2[t.prob], wr, N - col);
            }
            if (!W8 && p.out_g[t.prob] && nvalid > 0) {  // the pre-activation G and U as well (kept for the backward)
                const size_t r0 = static_cast<size_t>(t.out_row0 + wrow0) * N + col;
                stage_rows_f32(&stage[0][0], g, p.out_g[t.prob] + r0, N, nvalid, N - col);
                stage_rows_f32(&stage[0][0], u, p.out_u[t.prob] + r0, N, nvalid, N - col);
            }
            if (!valid) continue;
            __nv_bfloat16* dst = out + grow * N + col;
            __nv_bfloat16* dst_lo = out_lo ? out_lo + grow * N + col : nullptr;
            if (col + 32 <= N) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 pk, pk_lo;
                    uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
                    uint32_t* w_lo = reinterpret_cast<uint32_t*>(&pk_lo);
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const int i = q * 8 + h * 2;
                        const float h0 = silu_mul(__uint_as_float(g[i]), __uint_as_float(u[i]));
                        const float h1 = silu_mul(__uint_as_float(g[i + 1]), __uint_as_float(u[i + 1]));
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(h0, h1);
                        w[h] = *reinterpret_cast<uint32_t*>(&b2);
                        const float2 back = __bfloat1622float2(b2);
                        __nv_bfloat162 l2 = __floats2bfloat162_rn(h0 - back.x, h1 - back.y);
                        w_lo[h] = *reinterpret_cast<uint32_t*>(&l2);
                    }
                    reinterpret_cast<uint4*>(dst)[q] = pk;
                    if (dst_lo) reinterpret_cast<uint4*>(dst_lo)[q] = pk_lo;
                }
            } else {
                for (int i = 0; i < 32 && col + i < N; ++i) {
                    const float hv = silu_mul(__uint_as_float(g[i]), __uint_as_float(u[i]));
                    const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                    dst[i] = hb;
                    if (dst_lo) dst_lo[i] = __float2bfloat16_rn(hv - __bfloat162float(hb));
                }
            }
        }
    } else if (MODE == kGemmSwigluBwd) {
        // SwiGLU backward on D (this thread's row, 32 columns at a time).  The
        // G and U values of the next 32 columns are loaded while this chunk is
        // computed, so each chunk waits for at most one round trip to memory.
        const float g = (valid && p.row_scale[t.prob]) ? __ldg(p.row_scale[t.prob] + grow) : 1.0f;
        const float* Gr = p.bwd_G[t.prob] + grow * N;
        const float* Ur = p.bwd_U[t.prob] + grow * N;
        __nv_bfloat16* dGr = p.bwd_dGU[t.prob] + grow * 2 * N;
        __nv_bfloat16* Hr = p.bwd_Hb[t.prob] + grow * N;
        auto load_gu = [&](int col, float (&ga)[32], float (&ub)[32]) {
            const int nc = valid ? min(32, N - col) : 0;
            if (nc == 32) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 a4 = __ldg(reinterpret_cast<const float4*>(Gr + col) + q);
                    const float4 b4 = __ldg(reinterpret_cast<const float4*>(Ur + col) + q);
                    ga[4 * q] = a4.x, ga[4 * q + 1] = a4.y, ga[4 * q + 2] = a4.z, ga[4 * q + 3] = a4.w;
                    ub[4 * q] = b4.x, ub[4 * q + 1] = b4.y, ub[4 * q + 2] = b4.z, ub[4 * q + 3] = b4.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    ga[i] = i < nc ? __ldg(Gr + col + i) : 0.f;
                    ub[i] = i < nc ? __ldg(Ur + col + i) : 0.f;
                }
            }
        };
        float ga[32], ub[32];
        load_gu(t.n * BN, ga, ub);
        float part = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t v[32];
            __syncwarp();
            tmem_ld32(tacc + c0, v);
            tmem_ld_wait();
            const int col = t.n * BN + c0;
            float gn[32], un[32];
            if (c0 + 32 < BN) load_gu(col + 32, gn, un);
            if (valid && col < N) {
                const int nc = min(32, N - col);
                uint4 pg[4], pu[4], ph[4];
                swiglu_bwd_pack(ga, ub, v, nc, g, pg, pu, ph, part);
                store_bf16_row(pg, nc, dGr + col);
                store_bf16_row(pu, nc, dGr + N + col);
                store_bf16_row(ph, nc, Hr + col);
            }
            if (c0 + 32 < BN) {
#pragma unroll
                for (int i = 0; i < 32; ++i) ga[i] = gn[i], ub[i] = un[i];
            }
        }
        if (valid && p.bwd_dgp_part[t.prob]) p.bwd_dgp_part[t.prob][(size_t)t.n * p.bwd_dgp_ld[t.prob] + grow] = part;
    } else {
        // fp32 (or bf16) rows out: each 32x32 block of the warp's rows goes
        // through shared memory, written row by row (thread = row, 16-byte
        // chunks) and read back with 8 lanes per row, so that every store
        // instruction writes 4 whole row segments (measured against one 32-bit
        // store per row segment: the saved-activation backward's weight-gradient
        // GEMMs, 6.00 -> 5.85 ms per backward call on the Mixtral prefill shape;
        // a TMA store of each block, which shares the copy engine with the
        // operand loads, was slower: 6.50 ms).
        float* out = static_cast<float*>(p.out[t.prob]);
        float scale = 1.0f;
        if ((MODE == kGemmScale || MODE == kGemmScaleSplit) && valid && p.row_scale[t.prob] != nullptr)
            scale = __ldg(p.row_scale[t.prob] + grow);
        const int lane = threadIdx.x & 31;
        const int wrow0 = warp_row0 >= 0 ? warp_row0 : row_in_tile - lane;  // first tile row of this warp
        const int nvalid = min(warp_rows, t.rows_valid - wrow0);  // rows of this warp that exist
        // a K-grouped tile with an empty window computed nothing: its output is 0
        const bool computed = t.kb1 > t.kb0;
        // The next 32 accumulator columns are read from TMEM while this chunk's
        // rows are stored.  The 32 x 32 block in shared memory: row r's 16-byte
        // chunk j at float r * 32 + ((j ^ (r & 7)) << 2), so that both the
        // row-wise 16-byte writes and the 16-byte reads of 8 lanes per row hit
        // distinct banks.
        float* sb = &stage[0][0];
        auto sidx = [](int r, int c) { return r * 32 + ((((c >> 2) ^ (r & 7))) << 2) + (c & 3); };
        uint32_t v[32];
        __syncwarp();
        tmem_ld32(tacc, v);
        tmem_ld_wait();
#pragma unroll 1
        for (int c0 = 0; c0 < ncols; c0 += 32) {
            const int col = t.n * BN + col_lo + c0;
            const bool live = col < N && nvalid > 0;  // uniform across the warp
            if (live) {
                if (p.wscale1[t.prob])
                    apply_wscale32(v, p.wscale1[t.prob], static_cast<size_t>(t.g) * N + col, N - col);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4*>(sb + lane * 32 + ((j ^ (lane & 7)) << 2)) =
                        computed ? make_float4(scale * __uint_as_float(v[4 * j]), scale * __uint_as_float(v[4 * j + 1]),
                                               scale * __uint_as_float(v[4 * j + 2]), scale * __uint_as_float(v[4 * j + 3]))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            __syncwarp();
            const bool more = c0 + 32 < ncols;
            uint32_t vn[32];
            if (more) tmem_ld32(tacc + c0 + 32, vn);
            if (live) {
                const size_t row0 = (size_t)(t.out_row0 + wrow0);
                if (nvalid == 32 && col + 32 <= N && (N & 3) == 0) {
                    // 8 lanes per row, 4 rows per instruction: 16-byte reads, whole row segments out
                    const int rq = lane >> 3, jj = lane & 7;
                    float4 q[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = 4 * i + rq;
                        q[i] = *reinterpret_cast<const float4*>(sb + rr * 32 + ((jj ^ (rr & 7)) << 2));
                    }
                    if (p.out_bf16[t.prob]) {
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out[t.prob]) + row0 * N + col + 4 * jj;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            __nv_bfloat162 a = __floats2bfloat162_rn(q[i].x, q[i].y);
                            __nv_bfloat162 b = __floats2bfloat162_rn(q[i].z, q[i].w);
                            uint2 u;
                            u.x = *reinterpret_cast<uint32_t*>(&a);
                            u.y = *reinterpret_cast<uint32_t*>(&b);
                            *reinterpret_cast<uint2*>(dst + (size_t)(4 * i + rq) * N) = u;
                        }
                    } else {
                        float* dst = out + row0 * N + col + 4 * jj;
#pragma unroll
                        for (int i = 0; i < 8; ++i) *reinterpret_cast<float4*>(dst + (size_t)(4 * i + rq) * N) = q[i];
                    }
                } else {
                    const bool col_ok = col + lane < N;
                    if (p.out_bf16[t.prob]) {
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out[t.prob]) + row0 * N + col + lane;
                        for (int r = 0; r < nvalid; ++r)
                            if (col_ok) dst[(size_t)r * N] = __float2bfloat16_rn(sb[sidx(r, lane)]);
                    } else {
                        float* dst = out + row0 * N + col + lane;
                        for (int r = 0; r < nvalid; ++r)
                            if (col_ok) dst[(size_t)r * N] = sb[sidx(r, lane)];
                    }
                }
            }
            if (more) {
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = vn[i];
            }
            __syncwarp();  // the stage block is read before the next chunk overwrites it
        }
    }
}

// ------------------------------------------------------------------ kernel

template <int MODE, bool W8>
__global__ void __launch_bounds__(W8 ? W8_THREADS : NUM_THREADS, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using SC = StageCfg<MODE>;
    constexpr int NST = ring_stages<MODE, W8>();
    constexpr int SLOT = slot_bytes<MODE, W8>();
    constexpr int BOFF = slot_b_off<MODE, W8>();
    static_assert(!W8 || MODE == kGemmSwiGLU || MODE == kGemmScale, "FP8 weights: SwiGLU and Scale modes only");
    uint8_t* wide = smem + (size_t)NST * SLOT;  // FP8 variant: widened bf16 B tiles
    SmemTail& st = *reinterpret_cast<SmemTail*>(wide + (W8 ? (size_t)W8_WIDE * B_BYTES : 0));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int* abort_flag = &st.abort_flag;

    // ---- prologue: barriers, TMEM, tile prefix ----
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&st.full[s], 1);
            mbar_init(&st.empty[s], 1);
        }
        if (W8)
            for (int w = 0; w < W8_WIDE; ++w) {
                mbar_init(&st.wfull[w], 4);  // one arrival per converter warp
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
            prefetch_tmap(&p.tmA[q]);
            prefetch_tmap(&p.tmB1[q]);
            if (MODE == kGemmSwiGLU) prefetch_tmap(&p.tmB2[q]);
            if (SC::kSplit) prefetch_tmap(&p.tmA2[q]);
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&st.tmem_base)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // everything above touched no global memory: overlap it with the predecessor
    pdl_wait();
    if (warp == 2) {
        // tiles per group: ceil(rows / BM) * column blocks; warp-wide prefix sum
        for (int q = 0; q < 2; ++q) {
            int carry = 0;
            const int gb = q == 0 ? 0 : p.G[0];
            if (lane == 0) st.gbase[q] = gb;
            if (q < p.nprob) {
                const int ncb = (p.N[q] + out_cols_per_tile<MODE>() - 1) / out_cols_per_tile<MODE>();
                for (int base = 0; base < p.G[q]; base += 32) {
                    const int g = base + lane;
                    int tiles = 0;
                    if (g < p.G[q]) {
                        int lo = 0, hi = p.M[q];
                        if (p.offsets[q]) {
                            lo = p.offsets[q][g];
                            hi = p.offsets[q][g + 1];
                        }
                        if (lo < 0 || hi < lo || hi > p.a_rows[q]) {
                            record_status(p.status, kStatusBounds);
                            lo = hi = 0;
                        }
                        st.row0[gb + g] = lo;
                        st.rows[gb + g] = hi - lo;
                        tiles = ((hi - lo + BM - 1) / BM) * ncb * p.ksplit;
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
        // ---------------- TMA producer ----------------
        // Lane 0 arms each stage's barrier and loads B (and A when A is a plain
        // tile); when A rows are gathered, every lane loads 4 of the tile's
        // 128 rows with one gather4 per k-block.  FP8 weights: B is the raw
        // one-byte tile, widened later by the converter warps.
        int s = 0;
        uint32_t ph = 0;
        uint32_t issued_parity[NST];
        bool used[NST];
        for (int i = 0; i < NST; ++i) used[i] = false;
        bool dead = p.stall_producer != 0;
        for (int id = blockIdx.x; id < total_tiles && !dead; id += gridDim.x) {
            const Tile t = decode_tile<MODE>(st, p, id);
            const int b_row0 = (p.kbase[t.prob] ? 0 : t.g * p.N[t.prob]) + t.n * out_cols_per_tile<MODE>();
            const int32_t* gidx = p.a_gather[t.prob];
            int rows4[4] = {0, 0, 0, 0};
            if (gidx) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = lane * 4 + i;
                    int v = r < t.rows_valid ? __ldg(gidx + t.a_row0 + r) : 0;
                    if (v < 0 || v >= p.a_src_rows[t.prob]) {
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
                uint8_t* sa = smem + (size_t)s * SLOT;
                uint8_t* sb = sa + BOFF;
                if (lane == 0) {
                    // gathered A: only the groups of 4 rows that hold valid rows are
                    // loaded; the other rows of the tile are never stored
                    const uint32_t a_bytes = gidx ? (uint32_t)((t.rows_valid + 3) / 4) * 4 * (BK * 2) : A_BYTES;
                    const uint32_t b_bytes =
                        (MODE == kGemmPlain && p.mma_n != BN) ? (uint32_t)(p.mma_n * BK * 2) : (uint32_t)(SLOT - A_BYTES);
                    mbar_expect_tx(&st.full[s], b_bytes + a_bytes);
                    const int kc = t.k_off + kb * BK;
                    if (!W8 && MODE != kGemmSwiGLU && !SC::kSplit && p.b_mn) {  // B^T as 64-column blocks
                        uint64_t* bar = &st.full[s];
                        load_kblock_bmn(
                            p, t.prob, kb, t.a_row0, t.n * BN, t.g, BN / BK, sa, sb,
                            [bar](void* d, const CUtensorMap* tm, int c0, int c1, int c2) {
                                tma_load_3d(d, tm, c0, c1, c2, bar);
                            },
                            [bar](void* d, const CUtensorMap* tm, int c0, int c1) { tma_load_2d(d, tm, c0, c1, bar); });
                    } else {
                        if (!gidx) tma_load_2d(sa, &p.tmA[t.prob], kc, t.a_row0, &st.full[s]);
                        if (SC::kSplit) tma_load_2d(sa + A_BYTES, &p.tmA2[t.prob], kc, t.a_row0, &st.full[s]);
                        if (MODE == kGemmSwiGLU) {
                            tma_load_2d(sb, &p.tmB1[t.prob], kc, b_row0, &st.full[s]);
                            tma_load_2d(sb + (W8 ? F8_BYTES : B_BYTES) / 2, &p.tmB2[t.prob], kc, b_row0,
                                        &st.full[s]);
                        } else {
                            tma_load_2d(sb, &p.tmB1[t.prob], kc, b_row0, &st.full[s]);
                        }
                    }
                }
                if (gidx && lane * 4 < t.rows_valid)
                    tma_gather4(sa + lane * 4 * (BK * 2), &p.tmA[t.prob], kb * BK, rows4[0], rows4[1], rows4[2],
                                rows4[3], &st.full[s]);
                issued_parity[s] = ph;
                used[s] = true;
                if (++s == NST) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        // make sure no copy is still landing in shared memory before the CTA exits
        __syncwarp();
        if (lane == 0) {
            volatile int no_abort = 0;
            for (int i = 0; i < NST; ++i)
                if (used[i]) mbar_wait(&st.full[i], issued_parity[i], &no_abort, nullptr, kDrainLimitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const bool bmn = !W8 && MODE != kGemmSwiGLU && !SC::kSplit && p.b_mn;
            const int mn = MODE == kGemmPlain ? p.mma_n : BN;
            const uint32_t idesc_full = idesc_bf16_f32(BM, mn) | (bmn ? kIdescBMnMajor : 0u);
            const uint32_t idesc_m64 = idesc_bf16_f32(BM / 2, mn) | (bmn ? kIdescBMnMajor : 0u);
            int s = 0, w = 0;
            uint32_t ph = 0, pw = 0;
            int it = 0;
            bool dead = false;
            for (int id = blockIdx.x; id < total_tiles && !dead; id += gridDim.x, ++it) {
                const Tile t = decode_tile<MODE>(st, p, id);
                const uint32_t idesc = t.half ? idesc_m64 : idesc_full;
                const int acc = it & 1;
                const uint32_t use = static_cast<uint32_t>(it >> 1);
                if (!mbar_wait(&st.tmem_empty[acc], (use & 1u) ^ 1u, abort_flag, p.status, p.wait_limit_ns)) break;
                tc_fence_after();
                const uint32_t dtm = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait(&st.full[s], ph, abort_flag, p.status, p.wait_limit_ns)) {
                        dead = true;
                        break;
                    }
                    // FP8 weights: B comes from the widened tile, not the raw stage
                    if (W8 && !mbar_wait(&st.wfull[w], pw, abort_flag, p.status, p.wait_limit_ns)) {
                        dead = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)s * SLOT);
                    const uint32_t sb = W8 ? smem_u32(wide + (size_t)w * B_BYTES) : sa + BOFF;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint64_t bdesc = bmn ? sdesc_mn_sw128(sb + kk * UMMA_K * 128, BK * BK * 2)
                                                   : sdesc_k_sw128(sb + kk * UMMA_K * 2);
                        umma_bf16(dtm, sdesc_k_sw128(sa + kk * UMMA_K * 2), bdesc, idesc,
                                  (kb != t.kb0 || kk != 0) ? 1u : 0u);
                        if (SC::kSplit) umma_bf16(dtm, sdesc_k_sw128(sa + A_BYTES + kk * UMMA_K * 2), bdesc, idesc, 1u);
                    }
                    umma_commit(&st.empty[s]);
                    if (W8) {
                        umma_commit(&st.wempty[w]);
                        if (++w == W8_WIDE) {
                            w = 0;
                            pw ^= 1u;
                        }
                    }
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
        // ---------------- epilogue (warps 2..5) ----------------
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int row_in_tile = quarter * 32 + lane;
        int it = 0;
        for (int id = blockIdx.x; id < total_tiles; id += gridDim.x, ++it) {
            const Tile t = decode_tile<MODE>(st, p, id);
            const int acc = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            if (!mbar_wait(&st.tmem_full[acc], use & 1u, abort_flag, p.status, p.wait_limit_ns)) break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
            if (MODE != kGemmSwigluBwd && t.half)  // M = 64: rows 16q .. 16q + 15 in lanes 0-15 of quarter q
                epilogue_tile<MODE, W8>(p, t, tacc, lane < 16 ? quarter * 16 + lane : BM, st.stage[quarter], 0, BN, false,
                                    quarter * 16, 16);
            else
                epilogue_tile<MODE, W8>(p, t, tacc, row_in_tile, st.stage[quarter]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&st.tmem_empty[acc]);
        }
    } else if constexpr (W8) {
        // ---------------- converters (warps 6..9), FP8 weights ----------------
        // Per k-block: wait for the raw stage (A + one-byte B) to land and for
        // a free widened tile; each warp widens a quarter of the B tile, makes
        // its writes visible to the tensor cores' async proxy and arrives.
        // The raw stage itself is released by the MMA (it also reads A there).
        const int ctid = threadIdx.x - NUM_THREADS;  // 0..127
        int s = 0, w = 0;
        uint32_t ph = 0, pw = 0;
        bool dead = false;
        for (int id = blockIdx.x; id < total_tiles && !dead; id += gridDim.x) {
            const Tile t = decode_tile<MODE>(st, p, id);
            for (int kb = t.kb0; kb < t.kb1; ++kb) {
                const bool ok_w = mbar_wait(&st.wempty[w], pw ^ 1u, abort_flag, p.status, p.wait_limit_ns);
                const bool ok_raw = ok_w && mbar_wait(&st.full[s], ph, abort_flag, p.status, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, ok_raw)) {
                    dead = true;
                    break;
                }
                widen_b_tile(smem + (size_t)s * SLOT + BOFF, wide + (size_t)w * B_BYTES, ctid);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&st.wfull[w]);
                if (++w == W8_WIDE) {
                    w = 0;
                    pw ^= 1u;
                }
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
        // an aborted main loop may leave MMAs in flight: give them time to land
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {
        }
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
    }
    pdl_trigger();  // every epilogue store of this CTA precedes the teardown barrier
}

// ------------------------------------------------------- 2-SM (CTA pair) kernel
//
// For large expert segments: a cluster of two CTAs on two SMs computes one
// 256 x 256 tile with tcgen05.mma.cta_group::2 (M = 256: each CTA owns 128
// rows of A and of the accumulator; N = 256: each CTA holds half of the B
// tile and the pair's tensor cores share the halves).  Every SM therefore
// reads 32 KB of operands per 64-deep k-block instead of 48 KB, and the ring
// holds 6 stages instead of 4, which is what the 1-SM kernel lacks to keep
// its tensor cores fed.  Roles as in the 1-SM kernel; the leader CTA (rank 0)
// issues the MMAs, both CTAs load their own halves, both TMA streams signal
// the leader's stage barrier, MMA completion is multicast to both CTAs, and
// both CTAs' epilogue warps release the accumulator on the leader's barrier.

constexpr int PAIR_STAGE_BYTES = A_BYTES + B_BYTES / 2;  // this CTA's 128 rows of A + half of B
// The SwiGLU backward's epilogue reads two fp32 tensors (G, U) and writes
// three bf16 ones (dG, dU, H), each as large as its output: its ring keeps 4
// stages, and the freed shared memory stages those tiles for TMA (each
// epilogue warp: 2 slots of a 32 x 32 G box and a 32 x 32 U box, and one
// 32 x 32 box of each output, with 64-byte swizzle); the fp32 transpose
// buffer of the other epilogues is left out.
constexpr int GU_SLOT_BYTES = 32 * 32 * 4;
constexpr int GU_BYTES = 4 * 2 * 2 * GU_SLOT_BYTES;  // 4 warps x 2 slots x (G, U)
constexpr int OUT_BOX_BYTES = 32 * 32 * 2;
constexpr int OUT_BYTES = 4 * 3 * OUT_BOX_BYTES;  // 4 warps x (dG, dU, H)
// groups of both problems the CTA-pair SwiGLU backward takes (its shared
// memory holds no more); the launcher runs larger ones on single CTAs
constexpr int kPairBwdGroups = 512;
template <int MODE>
using PairTail =
    typename std::conditional<MODE == kGemmSwigluBwd, SmemTailT<kPairBwdGroups + 1>, SmemTail>::type;
template <int MODE>
constexpr int pair_stages() {
    return MODE == kGemmSwigluBwd ? 4 : kMaxRing;
}
template <int MODE>
constexpr size_t pair_gu_bytes() {
    return MODE == kGemmSwigluBwd ? (size_t)(GU_BYTES + OUT_BYTES) : 0;
}
template <int MODE>
constexpr size_t pair_smem_bytes() {
    return 1024 + (size_t)pair_stages<MODE>() * PAIR_STAGE_BYTES + pair_gu_bytes<MODE>() + sizeof(PairTail<MODE>);
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same variable in the leader CTA (rank 0)
__device__ __forceinline__ uint32_t leader_addr(const void* p) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(out) : "r"(smem_u32(p)));
    return out;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* tm, int c0, int c1, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* tm, int c0, int c1, int c2,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// arrive on the barrier at this offset in both CTAs of the pair
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)0x3)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// Pair tile: 256 rows of one group (128 per CTA) x 256 accumulator columns.
template <int MODE, class TailT>
__device__ __forceinline__ Tile decode_tile_pair(const TailT& st, const TcParams& p, int id, int rank) {
    Tile t;
    t.prob = (id < st.total[0]) ? 0 : 1;
    const int local = id - (t.prob ? st.total[0] : 0);
    const int gb = st.gbase[t.prob];
    const int* ts = st.tile_start + gb;
    int lo = 0, hi = p.G[t.prob] - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ts[mid] <= local) lo = mid;
        else hi = mid - 1;
    }
    t.g = lo;
    const int rows = st.rows[gb + lo];
    const int mt = (rows + 2 * BM - 1) / (2 * BM);
    const int r = local - ts[lo];
    t.ks = 0;
    t.n = r / mt;
    t.m = r - t.n * mt;
    // a last tile of at most 128 rows is an M = 128 MMA: 64 rows per CTA
    t.half = (p.pair_half && rows - t.m * 2 * BM <= BM) ? 1 : 0;
    const int per = t.half ? BM / 2 : BM;
    const int first = t.m * 2 * BM + rank * per;  // this CTA's first row inside the group
    t.a_row0 = st.row0[gb + lo] + first;
    t.rows_valid = min(per, rows - first);  // may be <= 0 for the upper CTA of a tail tile
    t.out_row0 = t.a_row0;
    t.k_off = 0;
    t.kb0 = 0;
    t.kb1 = k_blocks(p, t.prob);
    if (p.kbase[t.prob]) {  // K-grouped: shared A rows, the group's own K window
        t.out_row0 = t.g * p.M[t.prob] + first;
        t.k_off = __ldg(p.kbase[t.prob] + t.g);
        t.kb1 = (__ldg(p.klen[t.prob] + t.g) + BK - 1) / BK;
    }
    return t;
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_tc_pair_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int NST = pair_stages<MODE>();
    uint8_t* gu_stage = smem + (size_t)NST * PAIR_STAGE_BYTES;  // 1024-aligned (stages are 32 KB)
    PairTail<MODE>& st = *reinterpret_cast<PairTail<MODE>*>(gu_stage + pair_gu_bytes<MODE>());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_rank();
    const bool leader = rank == 0;
    const int cluster_id = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    volatile int* abort_flag = &st.abort_flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&st.full[s], 1);   // leader: one arrive (with the pair's bytes)
            mbar_init(&st.empty[s], 1);  // one multicast MMA commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&st.tmem_full[a], 1);
            mbar_init(&st.tmem_empty[a], 8);  // leader: 4 epilogue warps in each CTA
        }
        for (int w = 0; w < 4; ++w)
            for (int sl = 0; sl < 2; ++sl) mbar_init(&st.gu_full[w][sl], 1);
        st.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        for (int q = 0; q < p.nprob; ++q) {
            prefetch_tmap(&p.tmA[q]);
            prefetch_tmap(&p.tmB1[q]);
            if (MODE == kGemmSwiGLU) prefetch_tmap(&p.tmB2[q]);
            if (MODE == kGemmSwigluBwd) {
                prefetch_tmap(&p.tmG[q]);
                prefetch_tmap(&p.tmU[q]);
                prefetch_tmap(&p.tmdG[q]);
                prefetch_tmap(&p.tmdU[q]);
                prefetch_tmap(&p.tmH[q]);
            }
        }
    }
    if (warp == 1) {  // both CTAs of the pair allocate together
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&st.tmem_base)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    pdl_wait();
    if (warp == 2) {
        for (int q = 0; q < 2; ++q) {
            int carry = 0;
            const int gb = q == 0 ? 0 : p.G[0];
            if (lane == 0) st.gbase[q] = gb;
            if (q < p.nprob) {
                const int ncb = (p.N[q] + out_cols_per_tile<MODE>() - 1) / out_cols_per_tile<MODE>();
                for (int base = 0; base < p.G[q]; base += 32) {
                    const int g = base + lane;
                    int tiles = 0;
                    if (g < p.G[q]) {
                        int lo = 0, hi = p.M[q];
                        if (p.offsets[q]) {
                            lo = p.offsets[q][g];
                            hi = p.offsets[q][g + 1];
                        }
                        if (lo < 0 || hi < lo || hi > p.a_rows[q]) {
                            record_status(p.status, kStatusBounds);
                            lo = hi = 0;
                        }
                        st.row0[gb + g] = lo;
                        st.rows[gb + g] = hi - lo;
                        tiles = ((hi - lo + 2 * BM - 1) / (2 * BM)) * ncb;
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
    cluster_sync();  // the peer's barriers are initialised before anyone signals them
    tc_fence_after();
    const uint32_t tmem_base = st.tmem_base;
    const int total_tiles = st.total[0] + st.total[1];

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_parity[NST];
            bool used[NST];
            for (int i = 0; i < NST; ++i) used[i] = false;
            bool dead = p.stall_producer != 0;
            for (int id = cluster_id; id < total_tiles && !dead; id += nclusters) {
                const Tile t = decode_tile_pair<MODE>(st, p, id, rank);
                // this CTA's half of the B tile.  SwiGLU: 64 W1 (gate) rows and
                // the same 64 features' W3 (up) rows, so the tile's columns run
                // [G 0-63 | U 0-63 | G 64-127 | U 64-127] over its 128 features
                int b_row;
                const CUtensorMap* tmb = &p.tmB1[t.prob];
                if (MODE == kGemmSwiGLU)
                    b_row = t.g * p.N[t.prob] + t.n * (BN / 2) + rank * (BN / 4);
                else  // K-grouped problems share one B matrix
                    b_row = (p.kbase[t.prob] ? 0 : t.g * p.N[t.prob]) + t.n * BN + rank * (BN / 2);
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait(&st.empty[s], ph ^ 1u, abort_flag, p.status, p.wait_limit_ns)) {
                        dead = true;
                        break;
                    }
                    uint8_t* sa = smem + (size_t)s * PAIR_STAGE_BYTES;
                    uint8_t* sb = sa + A_BYTES;
                    const uint32_t full_leader = leader_addr(&st.full[s]);
                    if (leader) mbar_expect_tx(&st.full[s], 2 * PAIR_STAGE_BYTES);
                    if (MODE != kGemmSwiGLU && p.b_mn) {  // this CTA's 128 columns: two 64-column blocks
                        load_kblock_bmn(
                            p, t.prob, kb, t.a_row0, t.n * BN + rank * (BN / 2), t.g, BN / 2 / BK, sa, sb,
                            [full_leader](void* d, const CUtensorMap* tm, int c0, int c1, int c2) {
                                tma_load_3d_pair(d, tm, c0, c1, c2, full_leader);
                            },
                            [full_leader](void* d, const CUtensorMap* tm, int c0, int c1) {
                                tma_load_2d_pair(d, tm, c0, c1, full_leader);
                            });
                    } else {
                        tma_load_2d_pair(sa, &p.tmA[t.prob], t.k_off + kb * BK, t.a_row0, full_leader);
                        if (MODE == kGemmSwiGLU) {  // two 64-row boxes
                            tma_load_2d_pair(sb, &p.tmB1[t.prob], t.k_off + kb * BK, b_row, full_leader);
                            tma_load_2d_pair(sb + B_BYTES / 4, &p.tmB2[t.prob], t.k_off + kb * BK, b_row, full_leader);
                        } else {
                            tma_load_2d_pair(sb, tmb, t.k_off + kb * BK, b_row, full_leader);
                        }
                    }
                    issued_parity[s] = ph;
                    used[s] = true;
                    if (++s == NST) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // Copies of the leader land on its own barrier; wait for those.  The
            // peer's copies are covered by the leader's wait and the final
            // cluster barrier.
            if (leader) {
                volatile int no_abort = 0;
                for (int i = 0; i < NST; ++i)
                    if (used[i]) mbar_wait(&st.full[i], issued_parity[i], &no_abort, nullptr, kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const bool bmn = MODE != kGemmSwiGLU && p.b_mn;
            const uint32_t idesc_full = idesc_bf16_f32(2 * BM, BN) | (bmn ? kIdescBMnMajor : 0u);
            const uint32_t idesc_half = idesc_bf16_f32(BM, BN) | (bmn ? kIdescBMnMajor : 0u);
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool dead = false;
            for (int id = cluster_id; id < total_tiles && !dead; id += nclusters, ++it) {
                const Tile t = decode_tile_pair<MODE>(st, p, id, 0);
                const uint32_t idesc = t.half ? idesc_half : idesc_full;
                const int acc = it & 1;
                const uint32_t use = static_cast<uint32_t>(it >> 1);
                if (!mbar_wait(&st.tmem_empty[acc], (use & 1u) ^ 1u, abort_flag, p.status, p.wait_limit_ns)) break;
                tc_fence_after();
                const uint32_t dtm = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait(&st.full[s], ph, abort_flag, p.status, p.wait_limit_ns)) {
                        dead = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)s * PAIR_STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        umma_bf16_pair(dtm, sdesc_k_sw128(sa + kk * UMMA_K * 2),
                                       bmn ? sdesc_mn_sw128(sb + kk * UMMA_K * 128, BK * BK * 2)
                                           : sdesc_k_sw128(sb + kk * UMMA_K * 2),
                                       idesc, (kb != t.kb0 || kk != 0) ? 1u : 0u);
                    umma_commit_pair(&st.empty[s]);
                    if (++s == NST) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (dead) break;
                umma_commit_pair(&st.tmem_full[acc]);
            }
        }
    } else if constexpr (MODE == kGemmSwigluBwd) {
        // SwiGLU backward.  G and U of this warp's 32 rows come in by TMA, 32
        // columns per box, into two slots per tensor: the next chunk's loads
        // are in flight while one is computed, and a tile's first two chunks
        // are requested before its accumulator is ready.  dG, dU and H leave
        // through one 32 x 32 box each, stored by TMA, when all 32 rows of the
        // warp belong to the tile's group (a box must not spill into the next
        // group's rows); otherwise each thread stores its own row.
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // full 128-row tiles: TMEM lane = tile row
        float* gu = reinterpret_cast<float*>(gu_stage) + quarter * (GU_BYTES / 4 / 4);  // [slot][G | U][32][32]
        uint8_t* ob = gu_stage + GU_BYTES + quarter * (3 * OUT_BOX_BYTES);             // [dG | dU | H][32][64 B]
        uint64_t* gbar = st.gu_full[quarter];
        // 16-byte chunk j of this lane's output row, 64-byte swizzle
        const int o_row = lane * 64, o_sw = (lane >> 1) & 3;
        uint32_t seq = 0;  // chunks this warp has requested before the current tile
        int it = 0;
        bool ok = true;
        for (int id = cluster_id; ok && id < total_tiles; id += nclusters, ++it) {
            const Tile t = decode_tile_pair<MODE>(st, p, id, rank);
            const int r0 = t.out_row0 + quarter * 32;
            auto request = [&](int c) {  // chunk c of this tile into slot (seq + c) & 1
                if (lane == 0) {
                    const uint32_t slot = (seq + c) & 1u;
                    float* dst = gu + slot * (2 * 32 * 32);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(&gbar[slot], 2 * GU_SLOT_BYTES);
                    tma_load_2d(dst, &p.tmG[t.prob], t.n * BN + c * 32, r0, &gbar[slot]);
                    tma_load_2d(dst + 32 * 32, &p.tmU[t.prob], t.n * BN + c * 32, r0, &gbar[slot]);
                }
            };
            request(0);
            request(1);
            const int acc = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            if (!mbar_wait(&st.tmem_full[acc], use & 1u, abort_flag, p.status, p.wait_limit_ns)) break;
            tc_fence_after();
            const uint32_t tacc =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
            const int N = p.N[t.prob];
            const bool valid = row < t.rows_valid;
            const bool box_rows = t.rows_valid - quarter * 32 >= 32;  // (uniform across the warp)
            const size_t grow = static_cast<size_t>(t.out_row0 + row);
            const float g = (valid && p.row_scale[t.prob]) ? __ldg(p.row_scale[t.prob] + grow) : 1.0f;
            __nv_bfloat16* dGr = p.bwd_dGU[t.prob] + grow * 2 * N;
            __nv_bfloat16* Hr = p.bwd_Hb[t.prob] + grow * N;
            float part = 0.f;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                __syncwarp();
                tmem_ld32(tacc + c * 32, v);
                tmem_ld_wait();
                const uint32_t slot = (seq + c) & 1u;
                if (!mbar_wait(&gbar[slot], ((seq + c) >> 1) & 1u, abort_flag, p.status, p.wait_limit_ns)) {
                    ok = false;
                    break;
                }
                // box row `lane`: 16-byte chunk j sits at chunk j ^ (lane & 7) of its 128-byte row
                const float* gs = gu + slot * (2 * 32 * 32) + lane * 32;
                float ga[32], ub[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int o = (j ^ (lane & 7)) * 4;
                    const float4 a4 = *reinterpret_cast<const float4*>(gs + o);
                    const float4 b4 = *reinterpret_cast<const float4*>(gs + 32 * 32 + o);
                    ga[4 * j] = a4.x, ga[4 * j + 1] = a4.y, ga[4 * j + 2] = a4.z, ga[4 * j + 3] = a4.w;
                    ub[4 * j] = b4.x, ub[4 * j + 1] = b4.y, ub[4 * j + 2] = b4.z, ub[4 * j + 3] = b4.w;
                }
                __syncwarp();  // every lane has read the slot before it is requested again
                if (c + 2 < BN / 32) request(c + 2);
                const int col = t.n * BN + c * 32;
                if (col >= N) continue;  // (uniform across the warp)
                const int nc = min(32, N - col);
                uint4 pg[4], pu[4], ph[4];
                if (box_rows) {
                    swiglu_bwd_pack(ga, ub, v, nc, g, pg, pu, ph, part);
                    if (lane == 0) bulk_wait_read<0>();  // the previous boxes have left shared memory
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int o = o_row + ((j ^ o_sw) << 4);
                        *reinterpret_cast<uint4*>(ob + o) = pg[j];
                        *reinterpret_cast<uint4*>(ob + OUT_BOX_BYTES + o) = pu[j];
                        *reinterpret_cast<uint4*>(ob + 2 * OUT_BOX_BYTES + o) = ph[j];
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {  // columns past N are clipped by the tensor maps
                        tma_store_2d(&p.tmdG[t.prob], col, r0, ob);
                        tma_store_2d(&p.tmdU[t.prob], col, r0, ob + OUT_BOX_BYTES);
                        tma_store_2d(&p.tmH[t.prob], col, r0, ob + 2 * OUT_BOX_BYTES);
                        bulk_commit();
                    }
                } else if (valid) {
                    swiglu_bwd_pack(ga, ub, v, nc, g, pg, pu, ph, part);
                    store_bf16_row(pg, nc, dGr + col);
                    store_bf16_row(pu, nc, dGr + N + col);
                    store_bf16_row(ph, nc, Hr + col);
                }
            }
            if (!ok) break;
            seq += BN / 32;
            if (valid && p.bwd_dgp_part[t.prob]) p.bwd_dgp_part[t.prob][(size_t)t.n * p.bwd_dgp_ld[t.prob] + grow] = part;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(leader_addr(&st.tmem_empty[acc]));
        }
        if (lane == 0) bulk_wait<0>();  // every box is written before the CTA leaves
    } else {
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        int it = 0;
        for (int id = cluster_id; id < total_tiles; id += nclusters, ++it) {
            const Tile t = decode_tile_pair<MODE>(st, p, id, rank);
            const int acc = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            if (!mbar_wait(&st.tmem_full[acc], use & 1u, abort_flag, p.status, p.wait_limit_ns)) break;
            tc_fence_after();
            const uint32_t tacc =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
            // M = 128 tile: lanes 0-63 hold this CTA's 64 rows x the first 128
            // columns, lanes 64-127 the same rows x the other 128
            const int row = t.half ? (quarter & 1) * 32 + lane : row_in_tile;
            const int col_lo = t.half ? (quarter >> 1) * (BN / 2) : 0;
            epilogue_tile<MODE>(p, t, tacc, row, st.stage[quarter], col_lo, t.half ? BN / 2 : BN, MODE == kGemmSwiGLU);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(leader_addr(&st.tmem_empty[acc]));
        }
    }

    // ---- teardown: neither CTA leaves while its peer may still touch its
    // shared memory or barriers; then the pair frees its TMEM together ----
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {
        }
    }
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS));
    }
    pdl_trigger();
}

// ----------------------------------------------------------------- host side

template <int MODE, bool W8 = false>
cudaError_t launch_mode(const TcParams& prm, int grid, cudaStream_t s) {
    // the shared-memory opt-in is per device; remember it for the first 64 ordinals
    static uint64_t attr_set_mask = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (!bit || !(attr_set_mask & bit)) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_tc_kernel<MODE, W8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem_bytes<MODE, W8>()));
        if (e != cudaSuccess) return e;
        attr_set_mask |= bit;
    }
    launch_pdl(grouped_gemm_tc_kernel<MODE, W8>, dim3(grid), dim3(W8 ? W8_THREADS : NUM_THREADS),
               smem_bytes<MODE, W8>(), s, prm);
    return cudaGetLastError();
}

static_assert(smem_bytes<kGemmSwiGLU, true>() <= 232448, "FP8 SwiGLU kernel exceeds shared memory");
static_assert(smem_bytes<kGemmScale, true>() <= 232448, "FP8 Scale kernel exceeds shared memory");
static_assert(pair_smem_bytes<kGemmSwiGLU>() <= 232448 && pair_smem_bytes<kGemmScale>() <= 232448 &&
                  pair_smem_bytes<kGemmSwigluBwd>() <= 232448,
              "CTA-pair kernel exceeds shared memory");

template <int MODE>
cudaError_t launch_pair_mode(const TcParams& prm, int num_sms, cudaStream_t s) {
    static uint64_t attr_set_mask = 0;
    static int max_clusters[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (!bit || !(attr_set_mask & bit)) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_tc_pair_kernel<MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(pair_smem_bytes<MODE>()));
        if (e != cudaSuccess) return e;
        // persistent grid: only as many pairs as can be resident at once
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms / 2));
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = pair_smem_bytes<MODE>();
        int nc = 0;
        e = cudaOccupancyMaxActiveClusters(&nc, grouped_gemm_tc_pair_kernel<MODE>, &cfg);
        if (e != cudaSuccess || nc < 1) return e != cudaSuccess ? e : cudaErrorLaunchOutOfResources;
        if (dev < 64) max_clusters[dev] = nc;
        attr_set_mask |= bit;
    }
    const int nc = dev < 64 ? max_clusters[dev] : 1;
    const int clusters = nc < num_sms / 2 ? nc : num_sms / 2;
    launch_pdl(grouped_gemm_tc_pair_kernel<MODE>, dim3(2 * clusters), dim3(NUM_THREADS), pair_smem_bytes<MODE>(), s, prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_tc(int mode, const GemmProblem* probs, int nprob, int* status, int num_sms,
                           cudaStream_t s, int ksplit, bool pair) {
    if (nprob < 1 || nprob > 2 || ksplit < 1) return cudaErrorInvalidValue;
    TcParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.ksplit = ksplit;
    // rows of B per TMA box: half the tile for SwiGLU (the W1 / W3 halves) and,
    // in either mode, on a CTA pair (each CTA holds half of the N columns)
    // (SwiGLU on CTA pairs: two 64-row boxes per CTA, W1 and W3 of the same features)
    if (pair && mode == kGemmSwigluBwd && probs[0].G + (nprob > 1 ? probs[1].G : 0) > kPairBwdGroups + 1) pair = false;
    // a plain product with few columns (the router's logits): 64-column MMAs and B tiles
    const bool narrow = mode == kGemmPlain && !pair && nprob == 1 && probs[0].N <= 64 && !probs[0].b_mn &&
                        !probs[0].kbase && !probs[0].klen && !probs[0].a_gather;
    const int b_box = narrow ? 64 : (mode == kGemmSwiGLU && pair) ? BN / 4 : (mode == kGemmSwiGLU || pair) ? BN / 2 : BN;
    if (probs[0].G + (nprob > 1 ? probs[1].G : 0) > MAX_GROUPS + 1) return cudaErrorInvalidValue;
    for (int q = 0; q < nprob; ++q) {
        const GemmProblem& g = probs[q];
        if (g.G < 1 || g.G > MAX_GROUPS) return cudaErrorInvalidValue;
        if (q > 0 && g.b_mn != probs[0].b_mn) return cudaErrorInvalidValue;
        if (g.b_mn) {
            // B^T tiles of 64 K-rows x 64 columns; A plain, or split in two K parts
            if ((mode != kGemmPlain && mode != kGemmScale && mode != kGemmSwigluBwd) || g.a_gather || g.kbase || g.klen ||
                ksplit != 1 ||
                g.N % 8 != 0 || (g.kpart && (g.kpart % 8 != 0 || g.K != 2 * g.kpart || !g.B2)))
                return cudaErrorInvalidValue;
            const uint64_t N = (uint64_t)g.N, kp = (uint64_t)(g.kpart ? g.kpart : g.K);
            if (!make_tmap_3d(&prm.tmB1[q], g.B1, N, kp, (uint64_t)g.G, N * 2, kp * N * 2, BK, BK, 1))
                return cudaErrorInvalidValue;
            if (g.kpart) {
                if (!make_tmap_3d(&prm.tmB2[q], g.B2, N, kp, (uint64_t)g.G, N * 2, kp * N * 2, BK, BK, 1) ||
                    !make_tmap_3d(&prm.tmA[q], g.A, kp, 2, (uint64_t)g.a_rows, kp * 2, 2 * kp * 2, BK, 1, BM))
                    return cudaErrorInvalidValue;
                prm.kpart[q] = g.kpart;
            } else if (!make_tmap(&prm.tmA[q], g.A, g.a_rows, g.K, BM)) {
                return cudaErrorInvalidValue;
            }
            prm.b_mn = 1;
        } else {
            if (g.a_gather) {
                // A rows are gathered from a [a_src_rows][K] tensor, 4 rows per load
                if (!make_tmap(&prm.tmA[q], g.A, g.a_src_rows, g.K, 1)) return cudaErrorInvalidValue;
                prm.a_gather[q] = g.a_gather;
                prm.a_src_rows[q] = g.a_src_rows;
            } else if (!make_tmap(&prm.tmA[q], g.A, g.a_rows, g.K, BM)) {
                return cudaErrorInvalidValue;
            }
            // B rows: one [N][K] matrix per group, or one shared by every group (K-grouped)
            const int b_rows = g.kbase ? g.N : g.G * g.N;
            if (!make_tmap(&prm.tmB1[q], g.B1, b_rows, g.K, b_box)) return cudaErrorInvalidValue;
            if (mode == kGemmSwiGLU && !make_tmap(&prm.tmB2[q], g.B2, b_rows, g.K, b_box))
                return cudaErrorInvalidValue;
        }
        if (mode == kGemmScaleSplit && !make_tmap(&prm.tmA2[q], g.A2, g.a_rows, g.K, BM)) return cudaErrorInvalidValue;
        if (ksplit > 1) {
            // every slice needs at least one k-block
            if (ksplit > (g.K + BK - 1) / BK || g.part == nullptr) return cudaErrorInvalidValue;
            prm.part[q] = g.part;
            prm.part_cols[q] = mode == kGemmSwiGLU ? 2 * g.N : g.N;
        }
        if (mode == kGemmSwigluBwd) {
            if (!g.bwd_G || !g.bwd_U || !g.bwd_dGU || !g.bwd_Hb || ksplit != 1 || g.kbase || g.N % 8 != 0 ||
                (g.bwd_dgp_part && g.bwd_dgp_ld < g.a_rows))
                return cudaErrorInvalidValue;
            prm.bwd_G[q] = g.bwd_G;
            prm.bwd_U[q] = g.bwd_U;
            prm.bwd_dGU[q] = static_cast<__nv_bfloat16*>(g.bwd_dGU);
            prm.bwd_Hb[q] = static_cast<__nv_bfloat16*>(g.bwd_Hb);
            prm.bwd_dgp_part[q] = g.bwd_dgp_part;
            prm.bwd_dgp_ld[q] = g.bwd_dgp_ld;
            if (pair) {
                // N % 8 == 0: every row stride and dU's column offset are multiples of 16 bytes
                const uint64_t N = (uint64_t)g.N;
                __nv_bfloat16* dGU = static_cast<__nv_bfloat16*>(g.bwd_dGU);
                if ((reinterpret_cast<uintptr_t>(g.bwd_G) | reinterpret_cast<uintptr_t>(g.bwd_U) |
                     reinterpret_cast<uintptr_t>(g.bwd_dGU) | reinterpret_cast<uintptr_t>(g.bwd_Hb)) % 16 != 0 ||
                    !make_tmap_f32(&prm.tmG[q], g.bwd_G, g.a_rows, g.N) ||
                    !make_tmap_f32(&prm.tmU[q], g.bwd_U, g.a_rows, g.N) ||
                    !make_tmap_bf16_box32(&prm.tmdG[q], dGU, g.a_rows, g.N, 4 * N) ||
                    !make_tmap_bf16_box32(&prm.tmdU[q], dGU + N, g.a_rows, g.N, 4 * N) ||
                    !make_tmap_bf16_box32(&prm.tmH[q], g.bwd_Hb, g.a_rows, g.N, 2 * N))
                    return cudaErrorInvalidValue;
            }
        }
        if (g.out_g || g.out_u) {
            if (mode != kGemmSwiGLU || !g.out_g || !g.out_u || ksplit != 1 || g.N % 4 != 0) return cudaErrorInvalidValue;
            prm.out_g[q] = g.out_g;
            prm.out_u[q] = g.out_u;
        }
        if (g.out_bf16 && mode != kGemmScale && mode != kGemmScaleSplit) return cudaErrorInvalidValue;
        prm.offsets[q] = g.offsets;
        prm.out[q] = g.out;
        prm.out_bf16[q] = g.out_bf16;
        prm.out2[q] = g.out2;
        prm.row_scale[q] = g.row_scale;
        prm.G[q] = g.G;
        prm.M[q] = g.M;
        prm.N[q] = g.N;
        prm.K[q] = g.K;
        prm.a_rows[q] = g.a_rows;
        if (g.kbase || g.klen) {
            // 1-CTA: Plain mode; CTA pairs: Scale mode without row scales (the same product)
            const bool mode_ok = pair ? (mode == kGemmScale && !g.row_scale) : mode == kGemmPlain;
            if (!g.kbase || !g.klen || g.offsets || g.a_gather || ksplit != 1 || !mode_ok) return cudaErrorInvalidValue;
            prm.kbase[q] = g.kbase;
            prm.klen[q] = g.klen;
        }
    }
    prm.nprob = nprob;
    prm.status = status;
    prm.wait_limit_ns = kWaitLimitNs;
    prm.m64 = (pair || mode == kGemmSwigluBwd) ? 0 : 1;  // (the SwiGLU backward keeps 128-row tiles)
    prm.mma_n = narrow ? 64 : BN;
    // failure-path test switch: the producer issues no loads, so every CTA
    // with work gives up after a short bounded wait and reports MOE_ERR_TIMEOUT
    if (test_stall_gemm()) {
        prm.stall_producer = 1;
        prm.wait_limit_ns = kStallWaitLimitNs;
    }
    const int grid = num_sms > 0 ? num_sms : 148;
    if (pair) {
        // 2-SM tiles: plain A tiles only (no split-K, no gathered or split A)
        if (ksplit != 1 || prm.a_gather[0] || prm.a_gather[1]) return cudaErrorInvalidValue;
        // M = 128 tail tiles in every mode whose epilogue takes a column half
        prm.pair_half = mode != kGemmSwigluBwd ? 1 : 0;
        switch (mode) {
            case kGemmSwiGLU: return launch_pair_mode<kGemmSwiGLU>(prm, grid, s);
            case kGemmScale: return launch_pair_mode<kGemmScale>(prm, grid, s);
            case kGemmSwigluBwd: return launch_pair_mode<kGemmSwigluBwd>(prm, grid, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (mode) {
        case kGemmSwiGLU: return launch_mode<kGemmSwiGLU>(prm, grid, s);
        case kGemmScale: return launch_mode<kGemmScale>(prm, grid, s);
        case kGemmPlain: return launch_mode<kGemmPlain>(prm, grid, s);
        case kGemmSwigluBwd: return launch_mode<kGemmSwigluBwd>(prm, grid, s);
        case kGemmScaleSplit: return launch_mode<kGemmScaleSplit>(prm, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm_tc_w8(int mode, const GemmProblem* probs, int nprob, int* status, int num_sms,
                              cudaStream_t s, int ksplit) {
    if (nprob < 1 || nprob > 2 || ksplit < 1) return cudaErrorInvalidValue;
    if (mode != kGemmSwiGLU && mode != kGemmScale) return cudaErrorInvalidValue;
    TcParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.ksplit = ksplit;
    const int b_box = mode == kGemmSwiGLU ? BN / 2 : BN;
    if (probs[0].G + (nprob > 1 ? probs[1].G : 0) > MAX_GROUPS + 1) return cudaErrorInvalidValue;
    for (int q = 0; q < nprob; ++q) {
        const GemmProblem& g = probs[q];
        if (g.G < 1 || g.G > MAX_GROUPS || g.K % 16 != 0) return cudaErrorInvalidValue;
        if (!g.wscale1 || (mode == kGemmSwiGLU && !g.wscale2)) return cudaErrorInvalidValue;
        if (g.a_gather) {
            if (!make_tmap(&prm.tmA[q], g.A, g.a_src_rows, g.K, 1)) return cudaErrorInvalidValue;
            prm.a_gather[q] = g.a_gather;
            prm.a_src_rows[q] = g.a_src_rows;
        } else if (!make_tmap(&prm.tmA[q], g.A, g.a_rows, g.K, BM)) {
            return cudaErrorInvalidValue;
        }
        if (g.b_mn) return cudaErrorInvalidValue;
        if (!make_tmap_u8(&prm.tmB1[q], g.B1, g.G * g.N, g.K, b_box)) return cudaErrorInvalidValue;
        if (mode == kGemmSwiGLU && !make_tmap_u8(&prm.tmB2[q], g.B2, g.G * g.N, g.K, b_box))
            return cudaErrorInvalidValue;
        if (ksplit > 1) {
            if (ksplit > (g.K + BK - 1) / BK || g.part == nullptr) return cudaErrorInvalidValue;
            prm.part[q] = g.part;
            prm.part_cols[q] = mode == kGemmSwiGLU ? 2 * g.N : g.N;
        }
        if (g.out_bf16 && mode != kGemmScale) return cudaErrorInvalidValue;
        prm.offsets[q] = g.offsets;
        prm.out[q] = g.out;
        prm.out_bf16[q] = g.out_bf16;
        prm.out2[q] = g.out2;
        prm.row_scale[q] = g.row_scale;
        prm.wscale1[q] = g.wscale1;
        prm.wscale2[q] = g.wscale2;
        prm.G[q] = g.G;
        prm.M[q] = g.M;
        prm.N[q] = g.N;
        prm.K[q] = g.K;
        prm.a_rows[q] = g.a_rows;
    }
    prm.nprob = nprob;
    prm.status = status;
    prm.m64 = 1;
    prm.wait_limit_ns = kWaitLimitNs;
    if (test_stall_gemm()) {
        prm.stall_producer = 1;
        prm.wait_limit_ns = kStallWaitLimitNs;
    }
    const int grid = num_sms > 0 ? num_sms : 148;
    return mode == kGemmSwiGLU ? launch_mode<kGemmSwiGLU, true>(prm, grid, s) : launch_mode<kGemmScale, true>(prm, grid, s);
}

}  // namespace moe
