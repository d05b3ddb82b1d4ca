// gemm_simt.cu -- grouped expert GEMMs in IEEE fp32 on the CUDA cores.
//
// Same problems and epilogues as gemm_tc.cu (see there for the sources), for
// layers stored in fp32.  The tensor cores offer fp32 inputs only as TF32,
// whose 10-bit mantissa cannot meet an fp32 layer's tolerance, so fp32 layers
// use plain FMA tiles: 64x64 output tiles (32x64 when 64-row tiles would not
// give every SM one), K staged through shared memory 32 at a time (the next
// 32 loaded into registers while the current ones are multiplied), one 4x4
// register tile per thread (256 or 128 threads; two accumulator sets for the
// paired W1/W3 SwiGLU tile).  The up GEMM reads its token rows straight
// from x through the grouping's row order.  Every output still sums its K
// products in order.  Tiles are enumerated on the device from the group offsets; blocks
// beyond the real tile count exit at once.
#include "common.cuh"

namespace moe {
namespace {

constexpr int SB = 64;    // output columns of a tile (and its rows, unless a launch takes 32-row tiles)
constexpr int SK = 32;    // K slab
constexpr int SMAXG = kMaxExperts;

struct SimtParams {
    const float* A[2];
    const int32_t* a_gather[2];  // non-null: A row r is row a_gather[r] of A ([a_src_rows][K])
    int a_src_rows[2];
    const float* B1[2];
    const float* B2[2];
    const int32_t* offsets[2];
    float* out[2];
    const float* row_scale[2];
    int G[2], M[2], N[2], K[2], a_rows[2];
    int nprob;
};

// Rows [lo, hi) of group g of problem q: its offsets, or all M rows; a range
// that does not fit the A matrix is empty.
__device__ __forceinline__ void simt_grp_rows(const SimtParams& p, int q, int g, int& lo, int& hi) {
    lo = 0;
    hi = p.M[q];
    if (p.offsets[q]) {
        lo = __ldg(p.offsets[q] + g);
        hi = __ldg(p.offsets[q] + g + 1);
    }
    if (lo < 0 || hi < lo || hi > p.a_rows[q]) lo = hi = 0;
}

// TM: tile rows, 64 or 32 (4 TM threads: TM / 4 row groups x 16 column groups)
template <int MODE, int TM>
__global__ void __launch_bounds__(4 * TM) grouped_gemm_simt_kernel(const SimtParams p) {
    pdl_wait();
    __shared__ int s_start[2][SMAXG + 1];
    __shared__ int s_total[2];
    __shared__ __align__(16) float sA[SK][TM + 4];
    __shared__ __align__(16) float sB1[SK][SB + 4];
    __shared__ __align__(16) float sB2[SK][SB + 4];
    if (threadIdx.x == 0) {
        for (int q = 0; q < 2; ++q) {
            int run = 0;
            if (q < p.nprob) {
                const int ncb = (p.N[q] + SB - 1) / SB;
                for (int g = 0; g < p.G[q]; ++g) {
                    int lo, hi;
                    simt_grp_rows(p, q, g, lo, hi);
                    s_start[q][g] = run;
                    run += ((hi - lo + TM - 1) / TM) * ncb;
                }
            }
            s_total[q] = run;
        }
    }
    __syncthreads();
    for (int id = blockIdx.x; id < s_total[0] + s_total[1]; id += gridDim.x) {
        const int q = id < s_total[0] ? 0 : 1;
        const int local = id - (q ? s_total[0] : 0);
        int g = 0;
        while (g + 1 < p.G[q] && s_start[q][g + 1] <= local) ++g;
        int glo, ghi;
        simt_grp_rows(p, q, g, glo, ghi);
        const int mt = (ghi - glo + TM - 1) / TM;
        const int r = local - s_start[q][g];
        const int n = r / mt, m = r - (r / mt) * mt;
        const int row0 = glo + m * TM;
        const int rows_valid = min(TM, ghi - glo - m * TM);
        const int N = p.N[q], K = p.K[q];
        const int col0 = n * SB;
        const float* A = p.A[q];
        const float* B1 = p.B1[q] + (size_t)g * N * K;
        const float* B2 = (MODE == kGemmSwiGLU) ? p.B2[q] + (size_t)g * N * K : nullptr;
        const int tr = threadIdx.x / 16, tc = threadIdx.x % 16;
        float acc1[4][4] = {}, acc2[4][4] = {};
        // Loader role: thread t brings row t / 4 of the A slab and rows t / 4 +
        // TM j of the B1 (and B2) slabs (j < 64 / TM), the four-element groups
        // t % 4 and t % 4 + 4 of each slab row's eight (one 16-byte load each
        // when K % 4 == 0).  The next slab is loaded into these registers while
        // the current one is multiplied, so each slab waits for its loads at
        // most once.
        constexpr int NQ = SK / 16;  // four-element groups per thread and row
        constexpr int PB = SB / TM;  // B rows per thread
        const int lr = threadIdx.x >> 2, lq = threadIdx.x & 3;
        // 16-byte loads need K % 4 == 0 and 16-byte aligned operand bases (the
        // entry points reject other pointers and sizes; checked here as well so
        // that the kernel stays safe on its own)
        const uintptr_t bases = reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(p.B1[q]) |
                                (MODE == kGemmSwiGLU ? reinterpret_cast<uintptr_t>(p.B2[q]) : 0);
        const bool vec = (K & 3) == 0 && (bases & 15) == 0;
        const bool a_ok = lr < rows_valid;
        int a_src = row0 + (a_ok ? lr : 0);
        if (p.a_gather[q]) {  // rows straight from the token matrix, in expert order
            a_src = a_ok ? __ldg(p.a_gather[q] + a_src) : 0;
            if (a_src < 0 || a_src >= p.a_src_rows[q]) a_src = 0;
        }
        const float* a_row = A + (size_t)a_src * K;
        bool b_ok[PB];
        const float* b1_row[PB];
        const float* b2_row[PB];
#pragma unroll
        for (int j = 0; j < PB; ++j) {
            const int br = lr + TM * j;
            b_ok[j] = col0 + br < N;
            b1_row[j] = B1 + (size_t)(col0 + (b_ok[j] ? br : 0)) * K;
            b2_row[j] = (MODE == kGemmSwiGLU) ? B2 + (size_t)(col0 + (b_ok[j] ? br : 0)) * K : nullptr;
        }
        float ra[NQ][4], rb1[PB][NQ][4], rb2[PB][NQ][4];
        auto load4 = [&](const float* row, bool ok, int kg, float (&v)[4]) {
            if (vec && kg < K) {  // K % 4 == 0: the four elements are all in range or all out
                const float4 x = ok ? __ldg(reinterpret_cast<const float4*>(row + kg)) : make_float4(0.f, 0.f, 0.f, 0.f);
                v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = (ok && kg + e < K) ? __ldg(row + kg + e) : 0.f;
            }
        };
        auto fetch = [&](int k0) {
#pragma unroll
            for (int h = 0; h < NQ; ++h) {
                const int kg = k0 + (lq + 4 * h) * 4;
                load4(a_row, a_ok, kg, ra[h]);
#pragma unroll
                for (int j = 0; j < PB; ++j) {
                    load4(b1_row[j], b_ok[j], kg, rb1[j][h]);
                    if (MODE == kGemmSwiGLU) load4(b2_row[j], b_ok[j], kg, rb2[j][h]);
                }
            }
        };
        fetch(0);
        for (int k0 = 0; k0 < K; k0 += SK) {
#pragma unroll
            for (int h = 0; h < NQ; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int kk = (lq + 4 * h) * 4 + e;
                    sA[kk][lr] = ra[h][e];
#pragma unroll
                    for (int j = 0; j < PB; ++j) {
                        sB1[kk][lr + TM * j] = rb1[j][h][e];
                        if (MODE == kGemmSwiGLU) sB2[kk][lr + TM * j] = rb2[j][h][e];
                    }
                }
            __syncthreads();
            if (k0 + SK < K) fetch(k0 + SK);
#pragma unroll
            for (int kk = 0; kk < SK; ++kk) {
                const float4 a4 = *reinterpret_cast<const float4*>(&sA[kk][tr * 4]);
                const float4 b4 = *reinterpret_cast<const float4*>(&sB1[kk][tc * 4]);
                const float a[4] = {a4.x, a4.y, a4.z, a4.w};
                const float b1[4] = {b4.x, b4.y, b4.z, b4.w};
                float b2[4] = {0.f, 0.f, 0.f, 0.f};
                if (MODE == kGemmSwiGLU) {
                    const float4 c4 = *reinterpret_cast<const float4*>(&sB2[kk][tc * 4]);
                    b2[0] = c4.x, b2[1] = c4.y, b2[2] = c4.z, b2[3] = c4.w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc1[i][j] = fmaf(a[i], b1[j], acc1[i][j]);
                        if (MODE == kGemmSwiGLU) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
                    }
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = tr * 4 + i;
            if (rr >= rows_valid) continue;
            const size_t grow = (size_t)(row0 + rr);
            float scale = 1.f;
            if (MODE == kGemmScale && p.row_scale[q]) scale = p.row_scale[q][grow];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = col0 + tc * 4 + j;
                if (col >= N) continue;
                float v;
                if (MODE == kGemmSwiGLU) {
                    const float gt = acc1[i][j];
                    v = gt / (1.0f + expf(-gt)) * acc2[i][j];
                } else {
                    v = scale * acc1[i][j];
                }
                p.out[q][grow * N + col] = v;
            }
        }
    }
    __syncthreads();
    pdl_trigger();
}

}  // namespace

cudaError_t launch_gemm_simt_f32(int mode, const GemmProblem* probs, int nprob, cudaStream_t s) {
    if (nprob < 1 || nprob > 2) return cudaErrorInvalidValue;
    SimtParams prm{};
    long long tiles_max = 0;
    for (int q = 0; q < nprob; ++q) {
        const GemmProblem& g = probs[q];
        if (g.G < 1 || g.G > SMAXG) return cudaErrorInvalidValue;
        prm.A[q] = static_cast<const float*>(g.A);
        prm.a_gather[q] = g.a_gather;
        prm.a_src_rows[q] = g.a_src_rows;
        prm.B1[q] = static_cast<const float*>(g.B1);
        prm.B2[q] = static_cast<const float*>(g.B2);
        prm.offsets[q] = g.offsets;
        prm.out[q] = static_cast<float*>(g.out);
        prm.row_scale[q] = g.row_scale;
        prm.G[q] = g.G;
        prm.M[q] = g.M;
        prm.N[q] = g.N;
        prm.K[q] = g.K;
        prm.a_rows[q] = g.a_rows;
        const long long rows = g.offsets ? g.a_rows : g.M;
        tiles_max += ((rows + SB - 1) / SB + (g.offsets ? g.G : 0)) * ((g.N + SB - 1) / SB);
    }
    prm.nprob = nprob;
    if (tiles_max == 0) return cudaSuccess;
    // fewer 64-row tiles than SMs: 32-row tiles (half the work each, twice as many)
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const bool small = tiles_max < sms;
    if (small) {
        tiles_max = 0;
        for (int q = 0; q < nprob; ++q) {
            const GemmProblem& g = probs[q];
            const long long rows = g.offsets ? g.a_rows : g.M;
            tiles_max += ((rows + 31) / 32 + (g.offsets ? g.G : 0)) * ((g.N + SB - 1) / SB);
        }
    }
    const int grid = static_cast<int>(tiles_max < 65535 ? tiles_max : 65535);
    const dim3 block(small ? 128 : 256);
    switch (mode) {
        case kGemmSwiGLU:
            if (small) launch_pdl(grouped_gemm_simt_kernel<kGemmSwiGLU, 32>, dim3(grid), block, 0, s, prm);
            else launch_pdl(grouped_gemm_simt_kernel<kGemmSwiGLU, 64>, dim3(grid), block, 0, s, prm);
            break;
        case kGemmScale:
            if (small) launch_pdl(grouped_gemm_simt_kernel<kGemmScale, 32>, dim3(grid), block, 0, s, prm);
            else launch_pdl(grouped_gemm_simt_kernel<kGemmScale, 64>, dim3(grid), block, 0, s, prm);
            break;
        case kGemmPlain:
            if (small) launch_pdl(grouped_gemm_simt_kernel<kGemmPlain, 32>, dim3(grid), block, 0, s, prm);
            else launch_pdl(grouped_gemm_simt_kernel<kGemmPlain, 64>, dim3(grid), block, 0, s, prm);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace moe
