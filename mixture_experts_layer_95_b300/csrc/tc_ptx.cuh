// tc_ptx.cuh -- inline-PTX building blocks of the tensor-core kernels
// (mbarriers, TMA, tcgen05 MMA / TMEM, shared-memory descriptors, FP8
// widening) and the host-side tensor-map encoders.  Shared by gemm_tc.cu and
// gemm_decode.cu.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace tc {

constexpr int BK = 64;      // one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;  // K of one kind::f16 MMA
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr uint64_t kDrainLimitNs = 10000000ull;   // 10 ms to drain copies after an abort

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of `bar`.  Returns false when the CTA is
// aborting (another role gave up) or this wait ran out of time.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            *abort_flag = 1;
            record_status(status, kStatusTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int c0, int c1, int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Shared -> global tensor store of one box at (c0, c1); elements outside the
// tensor's extent are not written.  Completion is tracked per thread in bulk
// groups: bulk_commit() closes a group, bulk_wait_read<n>() waits until at most
// n groups still read shared memory, bulk_wait<n>() until their writes are done.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, int c0, int c1, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Four rows (r0..r3) x 64 columns starting at column c0 of a 2-D tensor whose
// map has a one-row box; lands in shared memory as four consecutive 128-byte
// rows, swizzled like a tiled load to the same address.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* tm, int c0, int r0, int r1, int r2, int r3,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row core groups 1024 bytes apart (SBO); LBO is unused for a
// swizzled K-major operand whose K extent per instruction (32 bytes) stays
// inside one swizzle row.  Bits 46-47 hold the descriptor version (1).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(16u >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;  // 128-byte swizzle
    return d;
}

// Shared-memory matrix descriptor: MN-major operand, 128-byte swizzle.  Each
// 128-byte row holds 64 consecutive M (or N) elements of one K index; 8
// K-rows form a 1024-byte swizzle atom and consecutive atoms along K are SBO
// = 1024 bytes apart; the next 64 M (N) elements start LBO = mn_block_bytes
// further on.  One kind::f16 MMA consumes 16 K-rows (two atoms), so the K
// steps of a 64-deep block advance the start address by 2048 bytes.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t mn_block_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((mn_block_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor bit: B is MN-major (transposed) in shared memory.
constexpr uint32_t kIdescBMnMajor = 1u << 16;

// Instruction descriptor for kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, dense, M x N.
constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                                  // D format: f32
           | (1u << 7)                                // A format: bf16
           | (1u << 10)                               // B format: bf16
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Instruction descriptor for kind::f8f6f4 with E4M3 A and B (format code 0
// for both), fp32 accumulator, both K-major, dense, M x N.  One MMA covers
// K = 32 codes, i.e. the same 32 bytes of a 128-byte swizzle row as a bf16
// kind::f16 MMA.
constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                                  // D format: f32
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[32]) {  // fills r[0..15]
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Two E4M3 codes, placed in bytes 1 and 3 of `sp`, -> two bf16 (low half
// first), exactly, with integer and bf16 ALU operations only (no conversion
// unit).  The 7 magnitude bits of a code, moved to bits 4..10 of a 16-bit
// lane, read as a bf16 whose value is the code's value times 2^-120 -- for
// normal codes (exponent field offset by 127 - 7) and for subnormal ones
// (m/8 * 2^-6 becomes the bf16 subnormal m/8 * 2^-126) alike; one bf16
// multiply by +-2^120 (the sign taken from the code) then gives the exact
// value, a normal bf16 with at most 4 significant bits.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t sp) {
    const uint32_t mag = (sp >> 4) & 0x07F007F0u;
    const uint32_t mul = (sp & 0x80008000u) | 0x7B807B80u;  // bf16 +-2^120 per lane
    const __nv_bfloat162 r =
        __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&mag), *reinterpret_cast<const __nv_bfloat162*>(&mul));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// One raw FP8 B tile (256 rows x 64 bytes, row-major, as the TMA unit wrote
// it) -> the bf16 K-major 128-byte-swizzled tile the MMA reads (row r at
// r * 128 bytes, its 16-byte chunk c at chunk c ^ (r % 8)).  128 threads,
// 16 chunks of 8 elements each; reads and writes are bank-conflict free.
__device__ __forceinline__ void widen_b_tile(const uint8_t* src, uint8_t* dst, int ctid) {
#pragma unroll 8
    for (int q = 0; q < 16; ++q) {
        const int idx = ctid + q * 128;
        const int r = idx >> 3, c = idx & 7;
        const uint2 raw = *reinterpret_cast<const uint2*>(src + r * BK + c * 8);
        uint4 out;
        out.x = e4m3x2_to_bf16x2(__byte_perm(raw.x, 0u, 0x1404));  // codes 0, 1
        out.y = e4m3x2_to_bf16x2(__byte_perm(raw.x, 0u, 0x3424));  // codes 2, 3
        out.z = e4m3x2_to_bf16x2(__byte_perm(raw.y, 0u, 0x1404));
        out.w = e4m3x2_to_bf16x2(__byte_perm(raw.y, 0u, 0x3424));
        *reinterpret_cast<uint4*>(dst + r * (BK * 2) + ((c ^ (r & 7)) << 4)) = out;
    }
}

// v[i] *= scale of weight row wrow + i (FP8 weights), for the 32 columns of
// one tcgen05.ld; rem = columns that exist from wrow on (>= 32: all).
__device__ __forceinline__ void apply_wscale32(uint32_t (&v)[32], const float* ws, size_t wrow, int rem) {
    if (rem >= 32) {
        const float4* p4 = reinterpret_cast<const float4*>(ws + wrow);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 sc = __ldg(p4 + q);
            v[4 * q] = __float_as_uint(__uint_as_float(v[4 * q]) * sc.x);
            v[4 * q + 1] = __float_as_uint(__uint_as_float(v[4 * q + 1]) * sc.y);
            v[4 * q + 2] = __float_as_uint(__uint_as_float(v[4 * q + 2]) * sc.z);
            v[4 * q + 3] = __float_as_uint(__uint_as_float(v[4 * q + 3]) * sc.w);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            v[i] = __float_as_uint(i < rem ? __uint_as_float(v[i]) * __ldg(ws + wrow + i) : 0.f);
    }
}

// ----------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// Encoded maps are remembered per host thread (the last kTmapCacheSize
// distinct argument sets), so a layer called again on the same buffers skips
// the driver's encoding: the map is a pure function of its arguments.
struct TmapKey {
    int dtype, rank, swizzle;
    const void* base;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    bool operator==(const TmapKey& o) const {
        if (dtype != o.dtype || rank != o.rank || swizzle != o.swizzle || base != o.base) return false;
        for (int i = 0; i < 3; ++i)
            if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
        return strides[0] == o.strides[0] && strides[1] == o.strides[1];
    }
};
constexpr int kTmapCacheSize = 64;
struct TmapCache {
    TmapKey key[kTmapCacheSize];
    CUtensorMap map[kTmapCacheSize];
    int n = 0, next = 0;
};

inline bool encode_cached(CUtensorMap* tm, CUtensorMapDataType dtype, int rank, const void* base,
                          const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                          CUtensorMapSwizzle swizzle) {
    thread_local TmapCache cache;
    TmapKey k{};
    k.dtype = static_cast<int>(dtype);
    k.rank = rank;
    k.swizzle = static_cast<int>(swizzle);
    k.base = base;
    for (int i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) k.strides[i] = strides[i];
    for (int i = 0; i < cache.n; ++i)
        if (cache.key[i] == k) {
            *tm = cache.map[i];
            return true;
        }
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(tm, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    cache.key[cache.next] = k;
    cache.map[cache.next] = *tm;
    cache.next = (cache.next + 1) % kTmapCacheSize;
    if (cache.n < kTmapCacheSize) ++cache.n;
    return true;
}

// 2-D bf16 tensor [rows][K] (K contiguous), box = 64 x box_rows, 128-byte swizzle.
inline bool make_tmap(CUtensorMap* tm, const void* base, int rows, int K, int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
    return encode_cached(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 3-D bf16 tensor with dims {d0 (contiguous), d1, d2} and byte strides s1, s2
// of dims 1 and 2; box = b0 x b1 x b2, 128-byte swizzle (b0 = 64).  Used for
// MN-major operand tiles (64 M/N elements x 64 K-rows of one group) and for
// K ranges padded per part (coordinates past a dim's extent read as zero).
inline bool make_tmap_3d(CUtensorMap* tm, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                         uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
    const cuuint64_t dims[3] = {d0, d1 > 0 ? d1 : 1, d2 > 0 ? d2 : 1};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {b0, b1, b2};
    return encode_cached(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 2-D fp32 tensor [rows][cols] (cols contiguous, a multiple of 4), box = 32
// columns (128 bytes) x 32 rows, 128-byte swizzle: 16-byte chunk j of box row r
// lands at r * 128 + ((j ^ (r & 7)) << 4) of a 1024-byte-aligned destination.
inline bool make_tmap_f32(CUtensorMap* tm, const void* base, int rows, int cols) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
    const cuuint32_t box[2] = {32, 32};
    return encode_cached(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 2-D bf16 tensor of `cols` columns per row, rows `row_bytes` apart (a multiple
// of 16), box = 32 columns (64 bytes) x 32 rows, 64-byte swizzle: 16-byte chunk
// j of box row r sits at r * 64 + ((j ^ ((r >> 1) & 3)) << 4) of a
// 512-byte-aligned shared buffer.
inline bool make_tmap_bf16_box32(CUtensorMap* tm, const void* base, int rows, int cols, uint64_t row_bytes) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {32, 32};
    return encode_cached(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

// 2-D one-byte (FP8 code) tensor [rows][K], box = box_cols x box_rows.  No
// swizzle (the converter warps re-lay the tile out for the MMA themselves),
// or, with sw128 and 128 columns, the 128-byte swizzle the MMA reads directly.
inline bool make_tmap_u8(CUtensorMap* tm, const void* base, int rows, int K, int box_rows, int box_cols = BK,
                         bool sw128 = false) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    return encode_cached(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box,
                         sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}


}  // namespace tc
}  // namespace moe
