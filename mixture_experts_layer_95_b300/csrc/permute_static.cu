// permute_static.cu -- moe_permute_static: the grouping step without a
// caller-provided workspace.
//
// moe_permute needs a little device scratch (one expert histogram per block of
// 64 tokens) and takes it from the caller's workspace.  Some callers cannot
// provide one: code that is handed only its input and output buffers (a
// plug-in slot with a fixed signature) or that runs under a runtime which
// forbids device allocation once it has started.  This entry point keeps that
// scratch in a fixed, file-scope device array instead, so such a caller only
// passes inputs and outputs.  It launches the same three kernels as
// moe_permute and produces the same outputs.
//
// The array is a device symbol: host code cannot use its name as a device
// address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it.  Under the
// CUDA runtime's lazy module loading that first call is also when the
// library's device code, the array included, is put on the device, so a
// caller that must not allocate later makes its first call at start-up.
#include <atomic>

#include "common.cuh"

// Room for one E-wide histogram per 64-token block: ceil(T / 64) * E int32
// values, at most 65,536 (256 KiB).
constexpr int kStaticScratchInts = 1 << 16;

// The scratch itself.  Every device that loads the library holds it until
// the process exits; every call on a device shares it.
static __device__ __align__(256) int32_t g_permute_scratch[kStaticScratchInts];

namespace moe {
namespace {

constexpr int kMaxDevices = 64;

// Device address of the scratch array on each device, filled on first use.
// Host threads may call concurrently: every writer stores the same address,
// and the atomics make those racing stores and loads well defined.
std::atomic<int32_t*> g_scratch_addr[kMaxDevices] = {};

int static_check(const moe_config* c) {
    if (!c) return MOE_ERR_NULL;
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_DTYPE;
    if (c->T < 0 || c->d < 8 || c->d % 8 || c->E < 1 || c->E > kMaxExperts || c->k < 1 || c->k > c->E ||
        c->k > 32 || (long long)c->T * c->k >= (1LL << 31))
        return MOE_ERR_SHAPE;
    if (c->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_SHAPE;  // token-choice grouping only
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_permute_static(const moe_config* cfg, const int32_t* topk_ids, const float* gates, const void* x,
                                  int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* sorted_token_ids,
                                  int32_t* slot_pos, float* gates_perm, void* x_perm, int32_t* n_dropped,
                                  moe_stream_t stream) {
    using namespace moe;
    const int rc = static_check(cfg);
    if (rc != MOE_OK) return rc;
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    const long long nblk = (c.T + kRouterTokensPerBlock - 1) / kRouterTokensPerBlock;
    if (nblk * c.E > kStaticScratchInts) return MOE_ERR_SHAPE;  // beyond the fixed scratch
    if (!topk_ids || !gates || !x || !counts || !kept || !offsets || !sorted_token_ids || !slot_pos ||
        !gates_perm || !x_perm || !n_dropped)
        return MOE_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x_perm) & 15u)) return MOE_ERR_ALIGN;

    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevices) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_DEVICE;
    int32_t* block_hist = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!block_hist) {
        // one-time set-up on this device (it is current here)
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        block_hist = static_cast<int32_t*>(p);
        g_scratch_addr[dev].store(block_hist, std::memory_order_relaxed);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // The histogram kernel rewrites every entry of block_hist that the scan
    // reads, so nothing in the array has to start at zero.  There is no
    // workspace status word here: out-of-range ids are skipped, not reported.
    GroupOut o{};
    o.counts = counts;
    o.kept = kept;
    o.offsets = offsets;
    o.sorted_token_ids = sorted_token_ids;
    o.slot_pos = slot_pos;
    o.gates_perm = gates_perm;
    o.n_dropped = n_dropped;
    const int chunk = kRouterTokensPerBlock;
    if (launch_group_hist(c.T, c.E, c.k, chunk, topk_ids, block_hist, nullptr, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_group_scan(c.T, c.E, c.k, chunk, c.capacity, topk_ids, gates, block_hist, o, nullptr, s) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_gather_rows(c.dtype, c.T, c.d, c.T * c.k, offsets + c.E, sorted_token_ids, x, x_perm, nullptr, s) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
