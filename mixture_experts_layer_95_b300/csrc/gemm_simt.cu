// gemm_simt.cu -- grouped expert GEMMs in IEEE fp32 on the CUDA cores.
//
// Same problems and epilogues as gemm_tc.cu (see there for the sources), for
// layers stored in fp32.  The tensor cores offer fp32 inputs only as TF32,
// whose 10-bit mantissa cannot meet an fp32 layer's tolerance, so fp32 layers
// use plain FMA tiles: 64x64 output tiles, K staged through shared memory 16
// at a time, 256 threads with a 4x4 register tile each (two accumulator sets
// for the paired W1/W3 SwiGLU tile).  Tiles are enumerated on the device from
// the group offsets; blocks beyond the real tile count exit at once.
#include "common.cuh"

namespace moe {
namespace {

constexpr int SB = 64;    // tile rows and output columns
constexpr int SK = 16;    // K slab
constexpr int SMAXG = kMaxExperts;

struct SimtParams {
    const float* A[2];
    const float* B1[2];
    const float* B2[2];
    const int32_t* offsets[2];
    float* out[2];
    const float* row_scale[2];
    int G[2], M[2], N[2], K[2], a_rows[2];
    int nprob;
};

template <int MODE>
__global__ void __launch_bounds__(256) grouped_gemm_simt_kernel(const SimtParams p) {
    pdl_wait();
    __shared__ int s_start[2][SMAXG + 1];
    __shared__ int s_row0[2][SMAXG];
    __shared__ int s_rows[2][SMAXG];
    __shared__ int s_total[2];
    __shared__ float sA[SK][SB + 4];
    __shared__ float sB1[SK][SB + 4];
    __shared__ float sB2[SK][SB + 4];
    if (threadIdx.x == 0) {
        for (int q = 0; q < 2; ++q) {
            int run = 0;
            if (q < p.nprob) {
                const int ncb = (p.N[q] + SB - 1) / SB;
                for (int g = 0; g < p.G[q]; ++g) {
                    int lo = 0, hi = p.M[q];
                    if (p.offsets[q]) {
                        lo = p.offsets[q][g];
                        hi = p.offsets[q][g + 1];
                    }
                    if (lo < 0 || hi < lo || hi > p.a_rows[q]) lo = hi = 0;
                    s_start[q][g] = run;
                    s_row0[q][g] = lo;
                    s_rows[q][g] = hi - lo;
                    run += ((hi - lo + SB - 1) / SB) * ncb;
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
        const int mt = (s_rows[q][g] + SB - 1) / SB;
        const int r = local - s_start[q][g];
        const int n = r / mt, m = r - (r / mt) * mt;
        const int row0 = s_row0[q][g] + m * SB;
        const int rows_valid = min(SB, s_rows[q][g] - m * SB);
        const int N = p.N[q], K = p.K[q];
        const int col0 = n * SB;
        const float* A = p.A[q];
        const float* B1 = p.B1[q] + (size_t)g * N * K;
        const float* B2 = (MODE == kGemmSwiGLU) ? p.B2[q] + (size_t)g * N * K : nullptr;
        const int tr = threadIdx.x / 16, tc = threadIdx.x % 16;
        float acc1[4][4] = {}, acc2[4][4] = {};
        for (int k0 = 0; k0 < K; k0 += SK) {
            for (int i = threadIdx.x; i < SB * SK; i += 256) {
                const int rr = i / SK, kk = i % SK;
                const int kg = k0 + kk;
                sA[kk][rr] = (rr < rows_valid && kg < K) ? A[(size_t)(row0 + rr) * K + kg] : 0.f;
                const bool bv = (col0 + rr < N) && kg < K;
                sB1[kk][rr] = bv ? B1[(size_t)(col0 + rr) * K + kg] : 0.f;
                if (MODE == kGemmSwiGLU) sB2[kk][rr] = bv ? B2[(size_t)(col0 + rr) * K + kg] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < SK; ++kk) {
                float a[4], b1[4], b2[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    a[i] = sA[kk][tr * 4 + i];
                    b1[i] = sB1[kk][tc * 4 + i];
                    if (MODE == kGemmSwiGLU) b2[i] = sB2[kk][tc * 4 + i];
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
    const int grid = static_cast<int>(tiles_max < 65535 ? tiles_max : 65535);
    switch (mode) {
        case kGemmSwiGLU: launch_pdl(grouped_gemm_simt_kernel<kGemmSwiGLU>, dim3(grid), dim3(256), 0, s, prm); break;
        case kGemmScale: launch_pdl(grouped_gemm_simt_kernel<kGemmScale>, dim3(grid), dim3(256), 0, s, prm); break;
        case kGemmPlain: launch_pdl(grouped_gemm_simt_kernel<kGemmPlain>, dim3(grid), dim3(256), 0, s, prm); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace moe
