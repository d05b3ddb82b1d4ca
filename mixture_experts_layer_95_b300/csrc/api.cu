// api.cu -- the C ABI of libmoe_b300.so (declared in include/moe_b300.h).
//
// Validates arguments on the host, carves the caller's workspace and enqueues
// the kernels of each step on the caller's stream.  No call allocates device
// memory, synchronises (except moe_last_device_status, which must) or keeps a
// pointer after returning.
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "common.cuh"

namespace moe {
namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxTopK = 32;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool use_gemm_router(const moe_config& c) { return !use_warp_router(c.E, c.d, c.dtype); }

size_t esize(const moe_config& c) { return c.dtype == MOE_BF16 ? 2 : 4; }

bool use_h_split(const moe_config& c) { return c.dtype == MOE_BF16 && c.h_split == 1; }

bool expert_choice(const moe_config& c) { return c.routing == MOE_ROUTE_EXPERT_CHOICE; }

// Bucket size C of expert-choice routing: capacity when positive, else
// floor(T k / E), clamped to [1, T].
int ec_bucket(const moe_config& c) {
    if (c.T == 0) return 0;
    long long C = c.capacity > 0 ? c.capacity : (long long)c.T * c.k / c.E;
    if (C < 1) C = 1;
    if (C > c.T) C = c.T;
    return (int)C;
}

// Rows of the permuted layout: T k routing decisions, or E C chosen pairs.
long long perm_rows(const moe_config& c) { return expert_choice(c) ? (long long)c.E * ec_bucket(c) : (long long)c.T * c.k; }

// Slots per token in slot_pos: k, or E under expert choice.
int slots_per_token(const moe_config& c) { return expert_choice(c) ? c.E : c.k; }

// Large expert segments (at least 512 rows per touched expert on average,
// bf16, a single bf16 H): both grouped GEMMs run on CTA pairs (2-SM
// tensor-core MMAs) with 256-row tiles, a segment's last tile shrinking to
// 128 rows (64 per SM) when that covers its remainder.  A pair reads 32 KB of
// operands per SM and k-block where a 1-SM 128-row tile reads 48 KB for the
// same MMA work.  Smaller segments keep the 1-SM kernel's 128-row tiles: at
// ~256 rows per expert (the DeepSeek-V3 shape) the pairs measured slower
// (8.06 against 7.51 ms per layer call, same box, same clocks).
constexpr int kPairMinRowsPerExpert = 512;
bool use_pair_gemm(const moe_config& c) {
    const long long n = perm_rows(c);
    const long long touched = n < c.E ? n : c.E;
    return c.dtype == MOE_BF16 && c.h_split == 0 && n >= kPairMinRowsPerExpert * touched;
}

// Decode-sized bf16 batches: at most 32 rows per touched expert on average.
bool decode_sized(const moe_config& c) {
    const long long n = perm_rows(c);
    const long long touched = n < c.E ? n : c.E;
    return c.dtype == MOE_BF16 && n <= 32 * touched;
}

// Decode-sized bf16 batches with a single bf16 H: both expert GEMMs put the
// weights on the MMA's M side (gemm_decode.cu), with 32 token rows per tile
// when the touched experts average at most 16 rows, else 64 (48 with FP8
// weights, decode_tile_rows).
bool use_decode_gemm(const moe_config& c) { return decode_sized(c) && !use_h_split(c); }

// The up GEMM gathers x rows itself (TMA gather4, 4 rows per load), so the
// layer skips the permuted copy: decode-sized batches, except that the
// decode GEMM with 64-row token tiles reads an explicit copy as plain tiles
// (16 gather4 loads per stage would limit its weight stream).
bool use_gather_a(const moe_config& c) {
    if (c.dtype == MOE_F32) return true;  // the CUDA-core up GEMM reads x rows through the row order
    if (!decode_sized(c)) return false;
    const long long n = perm_rows(c);
    const long long touched = n < c.E ? n : c.E;
    return !use_decode_gemm(c) || n <= 16 * touched;
}

int decode_tile_rows(const moe_config& c, bool w8 = false) {
    const long long n = perm_rows(c);
    const long long touched = n < c.E ? n : c.E;
    // FP8: a 64-row tile's hi and lo token codes (16 KB) leave room for four
    // 32 KB weight stages only; 48 rows keep five
    return n <= 16 * touched ? 32 : (w8 ? 48 : 64);
}

// ---- split-K for decode-sized batches ----------------------------------------
// When a grouped GEMM has too few output tiles to keep every SM streaming
// weights, each tile's K range is split into S slices (fp32 partials, summed
// in slice order afterwards).  S is a function of the configuration only (a
// nominal 148-SM B300), so the workspace size does not depend on the device.
constexpr int kNominalSms = 148;
constexpr int kMaxKSplit = 16;

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Smallest S whose waves are >= 90% full, else the fullest; 1 when the tile
// list already covers several waves.  max_s bounds S so that the slices'
// fp32 traffic stays small next to the weight bytes the split helps stream.
int choose_ksplit(long long est_tiles, int nk, long long max_s) {
    if (est_tiles <= 0 || est_tiles >= 4LL * kNominalSms || max_s < 2) return 1;
    int best = 1;
    double best_eff = 0.0;
    for (int S = 1; S <= kMaxKSplit && S <= nk && S <= max_s; ++S) {
        const long long units = est_tiles * S;
        const double eff = (double)units / ((double)ceil_div(units, kNominalSms) * kNominalSms);
        if (eff >= 0.9) return S;
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = S;
        }
    }
    return best;
}

struct Splits {
    int up = 1, down = 1;
    bool up_balanced = false;  // decode up GEMM: 2 slices cut where each CTA's equal share ends
};

// Tiles a grouped GEMM will have at least: every touched expert owns one or
// more 128-row tiles.
long long est_row_tiles(const moe_config& c) {
    const long long n = perm_rows(c);
    const long long touched = n < c.E ? n : c.E;
    const long long by_rows = ceil_div(n, 128);
    return by_rows > touched ? by_rows : touched;
}

// K slices of the router's logits GEMM (bf16, large E): enough 128-token x
// 256-expert tiles to fill the SMs; the slices are added by the softmax pass.
int router_ksplit(const moe_config& c) {
    if (c.dtype != MOE_BF16 || !use_gemm_router(c) || c.T == 0) return 1;
    const long long tiles = (long long)ceil_div(c.T, 128) * ceil_div(c.E, 256);
    return choose_ksplit(tiles, ceil_div(c.d, 64), 4);
}

Splits choose_splits_bf16(const moe_config& c) {
    Splits sp;
    if (c.dtype != MOE_BF16 || c.T == 0) return sp;
    const long long rt = est_row_tiles(c);
    const long long st = c.n_shared ? ceil_div(c.T, 128) : 0;
    const long long up = rt * ceil_div(c.d_ff, 128) + st * (c.n_shared ? ceil_div(c.d_ff_shared, 128) : 0);
    const long long dn = (rt + st) * ceil_div(c.d, 256);
    int nk_up = ceil_div(c.d, 64);
    int nk_dn = ceil_div(c.d_ff, 64);
    if (c.n_shared) nk_dn = nk_dn < ceil_div(c.d_ff_shared, 64) ? nk_dn : ceil_div(c.d_ff_shared, 64);
    // bytes: weights streamed vs one slice's fp32 partials written and read back
    const long long n = perm_rows(c);
    const long long touched = n < c.E ? n : c.E;
    const long long w_up = touched * 2LL * c.d_ff * c.d * 2 + (long long)c.n_shared * 2LL * c.d_ff_shared * c.d * 2;
    const long long p_up = 8LL * (n * 2 * c.d_ff + (long long)c.n_shared * c.T * 2 * c.d_ff_shared);
    const long long w_dn = touched * (long long)c.d * c.d_ff * 2 + (long long)c.n_shared * c.d * c.d_ff_shared * 2;
    const long long p_dn = 8LL * (n + (long long)c.n_shared * c.T) * c.d;
    sp.up = choose_ksplit(up, nk_up, w_up / (10 * p_up));
    sp.down = choose_ksplit(dn, nk_dn, w_dn / (10 * p_dn));
    return sp;
}

// With FP8 weights the decode GEMM's stages hold two k-blocks, so a K slice
// needs at least two; the workspace (sized for bf16) holds either choice.
bool use_decode_gemm(const moe_config& c);

Splits choose_splits(const moe_config& c, bool w8 = false) {
    Splits sp = choose_splits_bf16(c);
    // FP8 decode-sized up GEMMs with one to four waves of tiles and no shared
    // expert: instead of S uniform slices (whose tile count rarely divides
    // into whole waves), every CTA streams an equal contiguous share of all
    // tiles' k-blocks; a share of at least one tile leaves each tile in at
    // most two pieces, so two slices hold every partial sum.  (Measured on
    // one box: one token, FP8 0.0966 -> 0.0954 ms; with bf16 weights the
    // uniform slices stay faster, 0.1404 vs 0.1422 ms.)
    if (w8 && use_decode_gemm(c) && c.n_shared == 0 && sp.up > 1) {
        const long long up_tiles = est_row_tiles(c) * ceil_div(c.d_ff, 128);
        if (up_tiles >= kNominalSms && up_tiles < 4LL * kNominalSms) {
            sp.up = 2;
            sp.up_balanced = true;
            return sp;
        }
    }
    if (w8 && use_decode_gemm(c)) {
        const int up_max = ceil_div(c.d, 128), dn_max = ceil_div(c.d_ff, 128);
        const int dn_max_s = c.n_shared ? ceil_div(c.d_ff_shared, 128) : dn_max;
        sp.up = sp.up < up_max ? sp.up : up_max;
        sp.down = sp.down < dn_max ? sp.down : dn_max;
        sp.down = sp.down < dn_max_s ? sp.down : dn_max_s;
        if (sp.up < 1) sp.up = 1;
        if (sp.down < 1) sp.down = 1;
    }
    return sp;
}

// Byte offsets of every workspace region; `total` is the size.
struct Layout {
    size_t status, topk_ids, gates, p_part, block_hist, counts, kept, offsets, n_dropped, sorted, slot_pos,
        gates_perm, p_mean, f, L, logits, probs, x_perm, h, h_shared, h_lo, h_shared_lo, y_perm, y_shared, part_up,
        part_up_shared, part_dn, part_dn_shared, xq, xq_s, xsq, xsq_s, hq, hq_s, hsq, hsq_s, up_sync, up_sync_bytes,
        total;
};

// Output tiles of a decode-sized split-K up GEMM, at most: every touched
// group's rows in 32-row token tiles (one partial tile per group) times the
// 128-channel column blocks, plus the shared expert's.
size_t decode_up_tiles(const moe_config& c) {
    const long long n = perm_rows(c);
    const long long touched = n < c.E ? n : c.E;
    const long long routed = ((n + 31) / 32 + touched) * ((c.d_ff + 127) / 128);
    const long long shared = c.n_shared ? ((long long)(c.T + 31) / 32) * ((c.d_ff_shared + 127) / 128) : 0;
    return (size_t)(routed + shared);
}

Layout layout(const moe_config& c) {
    Layout l{};
    const size_t n = (size_t)perm_rows(c);
    const size_t nk = (size_t)c.T * c.k;  // token-choice routing outputs
    // histogram / p rows: the router's chunks, and moe_permute's 64-token chunks
    const size_t ch = (size_t)router_chunk(c.T, c.E, c.d, c.dtype);
    const size_t nblk_r = ((size_t)c.T + ch - 1) / ch;
    const size_t nblk_p = ((size_t)c.T + kRouterTokensPerBlock - 1) / kRouterTokensPerBlock;
    const size_t nblk = nblk_r > nblk_p ? nblk_r : nblk_p;
    const size_t E = (size_t)c.E;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes);
        return at;
    };
    l.status = take(16);  // [0] device status word, [1] grouping counter of the one-block-per-token router
    l.topk_ids = take(4 * nk);
    l.gates = take(4 * nk);
    l.p_part = take(4 * nblk * E);
    l.block_hist = take(4 * nblk * E);
    l.counts = take(4 * E);
    l.kept = take(4 * E);
    l.offsets = take(4 * (E + 1));
    l.n_dropped = take(4);
    l.sorted = take(4 * n);
    l.slot_pos = take(4 * (size_t)c.T * slots_per_token(c));
    l.gates_perm = take(4 * n);
    l.p_mean = take(4 * E);
    l.f = take(4 * E);
    l.L = take(4);
    l.logits = take(use_gemm_router(c) ? 4 * (size_t)router_ksplit(c) * c.T * E : 0);
    l.probs = take(expert_choice(c) ? 4 * (size_t)c.T * E : 0);
    l.x_perm = take(use_gather_a(c) ? 0 : n * c.d * esize(c));  // not needed when the up GEMM gathers x
    l.h = take(n * c.d_ff * esize(c));
    l.h_shared = take(c.n_shared ? (size_t)c.T * c.d_ff_shared * esize(c) : 0);
    const bool split = use_h_split(c);
    l.h_lo = take(split ? n * c.d_ff * esize(c) : 0);
    l.h_shared_lo = take(split && c.n_shared ? (size_t)c.T * c.d_ff_shared * esize(c) : 0);
    const size_t yb = c.yperm_bf16 ? 2 : 4;  // expert rows in bf16 or fp32
    l.y_perm = take(yb * n * c.d);
    l.y_shared = take(c.n_shared ? yb * (size_t)c.T * c.d : 0);
    const Splits sp = choose_splits(c);
    const size_t su = sp.up > 1 ? sp.up : 0, sd = sp.down > 1 ? sp.down : 0;
    l.part_up = take(4 * su * n * 2 * c.d_ff);
    l.part_up_shared = take(c.n_shared ? 4 * su * (size_t)c.T * 2 * c.d_ff_shared : 0);
    l.part_dn = take(4 * sd * n * c.d);
    l.part_dn_shared = take(c.n_shared ? 4 * sd * (size_t)c.T * c.d : 0);
    // decode-sized batches with FP8 weights: the tokens and H as E4M3 hi/lo
    // code pairs with a scale per row (the FP8 MMA takes FP8 on both sides)
    const bool q8 = use_decode_gemm(c);
    l.xq = take(q8 ? 2 * n * c.d : 0);  // token rows in expert order
    l.xq_s = take(q8 ? 4 * n : 0);
    l.xsq = take(q8 && c.n_shared ? 2 * (size_t)c.T * c.d : 0);  // every token, for the shared expert
    l.xsq_s = take(q8 && c.n_shared ? 4 * (size_t)c.T : 0);
    l.hq = take(q8 ? 2 * n * c.d_ff : 0);
    l.hq_s = take(q8 ? 4 * n : 0);
    l.hsq = take(q8 && c.n_shared ? 2 * (size_t)c.T * c.d_ff_shared : 0);
    l.hsq_s = take(q8 && c.n_shared ? 4 * (size_t)c.T : 0);
    // split-K decode up GEMM: per-output-tile slice counters (zeroed by
    // moe_workspace_init, zero again after every launch)
    l.up_sync_bytes = use_decode_gemm(c) && sp.up > 1 ? 4 * decode_up_tiles(c) : 0;
    l.up_sync = take(l.up_sync_bytes);
    l.total = off;
    return l;
}

// Backward-pass workspace: the forward layout, then these regions.
struct BLayout {
    size_t probs, xp, dyp, G, U, D, dGU, Hb, dgp, kbase, klen, dGT, dUT, HbT, xpT, dysT, dXp, dlog, R,
        wg_part, s_off, s_kbase, s_klen, Gs, Us, dGUs, Hbs, dGsT, dUsT, HbsT, xT, dyT, dXs, total;
    int ncols, ncols_s;
};


BLayout blayout(const moe_config& c) {
    BLayout b{};
    const size_t n = (size_t)c.T * c.k, E = c.E, F = c.d_ff, d = c.d, T = c.T, Fs = c.d_ff_shared;
    b.ncols = (int)(((long long)n + 64LL * c.E + 63) / 64 * 64);  // every expert's window, each rounded up to 64
    b.ncols_s = (int)((T + 63) / 64 * 64);
    const size_t nc = (size_t)b.ncols, ncs = (size_t)b.ncols_s;
    size_t off = layout(c).total;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes);
        return at;
    };
    b.probs = take(4 * T * E);
    b.xp = take(2 * n * d);
    b.dyp = take(2 * n * d);
    b.G = take(4 * n * F);
    b.U = take(4 * n * F);
    b.D = take(4 * ((F + 255) / 256) * ((n + 3) / 4 * 4));  // the gate-gradient partials of the D GEMM
    b.dGU = take(2 * n * 2 * F);
    b.Hb = take(2 * n * F);
    b.dgp = take(4 * ((n + 3) / 4 * 4));
    b.kbase = take(4 * E);
    b.klen = take(4 * E);
    b.dGT = take(2 * 2 * F * nc);  // dG^T windows, then dU^T (one transpose of the dG|dU rows writes both)
    b.dUT = b.dGT + 2 * F * nc;
    b.HbT = take(2 * F * nc);
    b.xpT = take(2 * d * nc);
    b.dysT = take(2 * d * nc);
    b.dXp = take(4 * n * d);
    b.dlog = take(4 * T * E);
    b.R = take(4 * T * d);
    b.wg_part = take(4 * (size_t)wgate_grad_split(c.E, c.d) * E * d);
    const bool sh = c.n_shared != 0;
    b.s_off = take(sh ? 8 : 0);
    b.s_kbase = take(sh ? 4 : 0);
    b.s_klen = take(sh ? 4 : 0);
    b.Gs = take(sh ? 4 * T * Fs : 0);
    b.Us = take(sh ? 4 * T * Fs : 0);
    b.dGUs = take(sh ? 2 * T * 2 * Fs : 0);
    b.Hbs = take(sh ? 2 * T * Fs : 0);
    b.dGsT = take(sh ? 2 * 2 * Fs * ncs : 0);
    b.dUsT = b.dGsT + 2 * Fs * ncs;
    b.HbsT = take(sh ? 2 * Fs * ncs : 0);
    b.xT = take(sh ? 2 * d * ncs : 0);
    b.dyT = take(sh ? 2 * d * ncs : 0);
    b.dXs = take(sh ? 4 * T * d : 0);
    b.total = off;
    return b;
}

template <typename P>
P* at(void* ws, size_t off) {
    return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_config(const moe_config* c) {
    if (!c) return MOE_ERR_NULL;
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_DTYPE;
    if (c->T < 0 || c->d < 8 || c->E < 1 || c->E > kMaxExperts || c->k < 1 || c->k > c->E || c->k > kMaxTopK ||
        c->d_ff < 8)
        return MOE_ERR_SHAPE;
    if ((long long)c->T * c->k >= (1LL << 31)) return MOE_ERR_SHAPE;
    if (c->n_shared != 0 && c->n_shared != 1) return MOE_ERR_SHAPE;
    if (c->n_shared == 1 && c->d_ff_shared < 8) return MOE_ERR_SHAPE;
    if (c->d % 8 || c->d_ff % 8 || (c->n_shared && c->d_ff_shared % 8)) return MOE_ERR_SHAPE;
    if (c->y_fp32 != 0 && c->y_fp32 != 1) return MOE_ERR_DTYPE;
    if (c->h_split != 0 && c->h_split != 1) return MOE_ERR_DTYPE;
    if (c->routing != MOE_ROUTE_TOKEN_CHOICE && c->routing != MOE_ROUTE_EXPERT_CHOICE) return MOE_ERR_SHAPE;
    if (c->yperm_bf16 != 0 && (c->yperm_bf16 != 1 || c->dtype != MOE_BF16)) return MOE_ERR_DTYPE;
    if (c->routing == MOE_ROUTE_EXPERT_CHOICE) {
        if ((long long)c->T * c->E >= (1LL << 31)) return MOE_ERR_SHAPE;
        if ((long long)c->E * ec_bucket(*c) >= (1LL << 31)) return MOE_ERR_SHAPE;
    }
    // the grouped GEMM tile list holds at most kMaxExperts row groups
    return MOE_OK;
}

int check_ws(const moe_config* c, const void* ws, size_t ws_bytes) {
    if (!ws) return MOE_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(ws) % kAlign) return MOE_ERR_WORKSPACE;
    if (ws_bytes < layout(*c).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

// Device capability (10.3) and SM count, cached per ordinal.
int device_sms(int* sms_out) {
    static int cache_sms[64] = {0};
    static int cache_ok[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 64 && cache_ok[dev]) {
        *sms_out = cache_sms[dev];
        return cache_ok[dev] > 0 ? MOE_OK : MOE_ERR_DEVICE;
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    const bool ok = (major == 10 && minor == 3);
    if (dev < 64) {
        cache_sms[dev] = sms;
        cache_ok[dev] = ok ? 1 : -1;
    }
    *sms_out = sms;
    return ok ? MOE_OK : MOE_ERR_DEVICE;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ---- diagnostics: stage events and launch count ----
constexpr int kStageEvents = 12;
thread_local cudaEvent_t g_stage_events[kStageEvents] = {};
thread_local int g_stage_n = 0;
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_test_stall{0};

enum Stage { kStageRouter = 0, kStageScan = 1, kStageGather = 2, kStageUp = 3, kStageDown = 4, kStageCombine = 5 };

void stage_mark(int idx, cudaStream_t s) {
    if (idx >= g_stage_n || !g_stage_events[idx]) return;
    // under stream capture the event becomes a record node of the graph, so
    // that every replay records it (a plain record would only order the capture)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(g_stage_events[idx], s, cudaEventRecordExternal);
    else
        cudaEventRecord(g_stage_events[idx], s);
}

// Records the stage's start event on construction and its stop event on scope exit.
struct StageScope {
    int stage;
    cudaStream_t stream;
    StageScope(int st, cudaStream_t s) : stage(st), stream(s) { stage_mark(2 * stage, stream); }
    ~StageScope() { stage_mark(2 * stage + 1, stream); }
};

#define MOE_TRY(expr)               \
    do {                            \
        const int _rc = (expr);     \
        if (_rc != MOE_OK) return _rc; \
    } while (0)

#define MOE_CUDA(expr) MOE_TRY(cuda_rc(expr))

// One kernel launch: fails with MOE_ERR_CUDA, counts successful launches.
#define MOE_LAUNCH(expr)                                        \
    do {                                                        \
        if ((expr) != cudaSuccess) return MOE_ERR_CUDA;         \
        g_launches.fetch_add(1, std::memory_order_relaxed);     \
    } while (0)

// Router: logits, softmax, top-k (k = c.k), per-block partial sums of p and
// id histograms.  Expert choice calls it with k = 0 (softmax only) and a
// probs [T][E] output.
int enqueue_route(const moe_config& c, const Layout& L, void* ws, const void* x, const void* w_gate,
                  const float* logit_bias, const float* select_bias, int32_t* topk_ids, float* gates,
                  int32_t* block_hist, int sms, cudaStream_t s, int k, float* probs = nullptr) {
    float* p_part = at<float>(ws, L.p_part);
    StageScope scope(kStageRouter, s);
    if (use_split_d_router(c.T, c.E)) {
        MOE_LAUNCH(launch_router_split_d(c.dtype, c.T, c.d, c.E, k, x, w_gate, logit_bias, select_bias,
                                         c.renormalize, topk_ids, gates, p_part, block_hist, s, probs));
        return MOE_OK;
    }
    if (!use_gemm_router(c)) {
        MOE_LAUNCH(launch_router_warp(c.dtype, c.T, c.d, c.E, k, x, w_gate, logit_bias, select_bias, c.renormalize,
                                    topk_ids, gates, p_part, block_hist, s, probs));
        return MOE_OK;
    }
    float* logits = at<float>(ws, L.logits);
    GemmProblem g{};
    g.A = x;
    g.a_rows = c.T;
    g.B1 = w_gate;
    g.G = 1;
    g.M = c.T;
    g.N = c.E;
    g.K = c.d;
    g.out = logits;
    const int rs = router_ksplit(c);
    if (rs > 1) g.part = logits;  // K slices [rs][T][E]
    if (c.dtype == MOE_BF16)
        MOE_LAUNCH(launch_gemm_tc(kGemmPlain, &g, 1, at<int>(ws, L.status), sms, s, rs));
    else
        MOE_LAUNCH(launch_gemm_simt_f32(kGemmPlain, &g, 1, s));
    MOE_LAUNCH(launch_router_from_logits(c.T, c.E, k, logits, logit_bias, select_bias, c.renormalize, topk_ids,
                                       gates, p_part, block_hist, s, probs, rs));
    return MOE_OK;
}

// Router, softmax, top-k, then the grouping into `o` (statistics too when
// o.p_part is set).  Decode-sized batches (the one-block-per-token router)
// group inside the router launch: its last block to finish does it, counted
// in on the workspace word after the status word.  Otherwise the grouping
// scan follows as its own launch.
int enqueue_route_group(const moe_config& c, const Layout& L, void* ws, const void* x, const void* w_gate,
                        const float* logit_bias, const float* select_bias, int32_t* topk_ids, float* gates,
                        const GroupOut& o, int sms, cudaStream_t s, float* probs = nullptr) {
    int* status = at<int>(ws, L.status);
    int32_t* block_hist = at<int32_t>(ws, L.block_hist);
    if (use_split_d_router(c.T, c.E)) {
        StageScope scope(kStageRouter, s);
        MOE_LAUNCH(launch_router_split_d(c.dtype, c.T, c.d, c.E, c.k, x, w_gate, logit_bias, select_bias,
                                         c.renormalize, topk_ids, gates, at<float>(ws, L.p_part), block_hist, s, probs,
                                         &o, c.capacity, reinterpret_cast<unsigned int*>(status + 1), status));
        return MOE_OK;
    }
    MOE_TRY(enqueue_route(c, L, ws, x, w_gate, logit_bias, select_bias, topk_ids, gates, block_hist, sms, s, c.k,
                          probs));
    const int chunk = router_chunk(c.T, c.E, c.d, c.dtype);
    StageScope scope(kStageScan, s);
    MOE_LAUNCH(launch_group_scan(c.T, c.E, c.k, chunk, c.capacity, topk_ids, gates, block_hist, o, status, s));
    return MOE_OK;
}

// Expert-choice routing + grouping: softmax rows into probs, then every
// expert's bucket.  counts / kept / n_empty nullable.
int enqueue_route_ec(const moe_config& c, const Layout& L, void* ws, const void* x, const void* w_gate,
                     const float* logit_bias, float* probs, int32_t* sorted, float* gates_perm, int32_t* slot_pos,
                     int32_t* counts, int32_t* kept, int32_t* offsets, int32_t* n_empty, int sms, cudaStream_t s) {
    MOE_TRY(enqueue_route(c, L, ws, x, w_gate, logit_bias, nullptr, nullptr, nullptr, nullptr, sms, s, 0, probs));
    StageScope scope(kStageScan, s);
    MOE_LAUNCH(launch_ec_select(c.T, c.E, ec_bucket(c), probs, sorted, gates_perm, slot_pos, counts, kept, offsets,
                                n_empty, s));
    return MOE_OK;
}

// Both expert GEMMs.  With split-K on the down GEMM, reduce_down = true sums
// the slices into y_perm / y_shared (moe_expert_ffn); otherwise the slices are
// left in the workspace for the split-aware combine (moe_forward).
int enqueue_ffn(const moe_config& c, const Layout& L, void* ws, const void* x_perm, const int32_t* offsets,
                const float* gates_perm, const void* w1, const void* w3, const void* w2, const void* x,
                const void* ws1, const void* ws3, const void* ws2, void* y_perm, void* y_shared, int sms,
                cudaStream_t s, bool reduce_down, const int32_t* gather_idx, const moe_fp8_weights* w8 = nullptr) {
    const Splits sp = choose_splits(c, w8 != nullptr);
    const int n = (int)perm_rows(c);
    void* h = at<void>(ws, L.h);
    void* hs = at<void>(ws, L.h_shared);
    const bool split = use_h_split(c);
    void* h_lo = split ? at<void>(ws, L.h_lo) : nullptr;
    void* hs_lo = split && c.n_shared ? at<void>(ws, L.h_shared_lo) : nullptr;
    GemmProblem up[2] = {}, down[2] = {};
    up[0].A = x_perm;
    up[0].a_rows = n;
    if (gather_idx) {  // rows come straight from x, in permuted order
        up[0].A = x;
        up[0].a_gather = gather_idx;
        up[0].a_src_rows = c.T;
    }
    up[0].B1 = w1;
    up[0].B2 = w3;
    up[0].offsets = offsets;
    up[0].G = c.E;
    up[0].N = c.d_ff;
    up[0].K = c.d;
    up[0].out = h;
    up[0].out2 = h_lo;
    down[0].A = h;
    down[0].A2 = h_lo;
    down[0].a_rows = n;
    down[0].B1 = w2;
    down[0].offsets = offsets;
    down[0].G = c.E;
    down[0].N = c.d;
    down[0].K = c.d_ff;
    down[0].out = y_perm;
    down[0].out_bf16 = c.yperm_bf16;
    down[0].row_scale = gates_perm;
    int np = 1;
    if (c.n_shared) {
        up[1].A = x;
        up[1].a_rows = c.T;
        up[1].B1 = ws1;
        up[1].B2 = ws3;
        up[1].G = 1;
        up[1].M = c.T;
        up[1].N = c.d_ff_shared;
        up[1].K = c.d;
        up[1].out = hs;
        up[1].out2 = hs_lo;
        down[1].A = hs;
        down[1].A2 = hs_lo;
        down[1].a_rows = c.T;
        down[1].B1 = ws2;
        down[1].G = 1;
        down[1].M = c.T;
        down[1].N = c.d;
        down[1].K = c.d_ff_shared;
        down[1].out = y_shared;
        down[1].out_bf16 = c.yperm_bf16;
        np = 2;
    }
    if (sp.up > 1) {
        up[0].part = at<float>(ws, L.part_up);
        up[1].part = at<float>(ws, L.part_up_shared);
    }
    if (sp.down > 1) {
        down[0].part = at<float>(ws, L.part_dn);
        down[1].part = at<float>(ws, L.part_dn_shared);
    }
    if (w8) {  // FP8 codes in place of the bf16 weights, plus their row scales
        up[0].B1 = w8->w1;
        up[0].B2 = w8->w3;
        up[0].wscale1 = w8->s1;
        up[0].wscale2 = w8->s3;
        down[0].B1 = w8->w2;
        down[0].wscale1 = w8->s2;
        up[1].B1 = w8->ws1;
        up[1].B2 = w8->ws3;
        up[1].wscale1 = w8->ss1;
        up[1].wscale2 = w8->ss3;
        down[1].B1 = w8->ws2;
        down[1].wscale1 = w8->ss2;
    }
    int* status = at<int>(ws, L.status);
    // FP8 decode GEMMs read the tokens (and H) as E4M3 hi/lo codes: x -> xq
    // (rows already in expert order, so the up GEMM loads plain tiles instead
    // of gathering twice as many code rows) and xsq (the shared expert's) here,
    // H -> hq between the two GEMMs
    const bool q8 = w8 && use_decode_gemm(c);
    uint8_t* xq = q8 ? at<uint8_t>(ws, L.xq) : nullptr;
    uint8_t* xsq = q8 && c.n_shared ? at<uint8_t>(ws, L.xsq) : nullptr;
    uint8_t* hq = q8 ? at<uint8_t>(ws, L.hq) : nullptr;
    uint8_t* hsq = q8 && c.n_shared ? at<uint8_t>(ws, L.hsq) : nullptr;
    if (q8 && !gather_idx) return MOE_ERR_SHAPE;  // the fused layer always passes the expert order
    if (q8) {
        up[0].A = xq;
        up[0].A2 = xq + (size_t)n * c.d;
        up[0].a_scale = at<float>(ws, L.xq_s);
        up[0].a_gather = nullptr;
        up[0].a_rows = n;
        if (c.n_shared) {
            up[1].A = xsq;
            up[1].A2 = xsq + (size_t)c.T * c.d;
            up[1].a_scale = at<float>(ws, L.xsq_s);
        }
        for (int q = 0; q < np; ++q) {
            down[q].A = q == 0 ? hq : hsq;
            down[q].A2 = q == 0 ? hq + (size_t)n * c.d_ff : hsq + (size_t)c.T * c.d_ff_shared;
            down[q].a_scale = at<float>(ws, q == 0 ? L.hq_s : L.hsq_s);
        }
    }
    if (q8) {  // token rows for the up GEMM, timed with the gather step
        StageScope scope(kStageGather, s);
        MOE_LAUNCH(launch_split_e4m3(n, c.d, x, c.T, gather_idx, offsets + c.E, xq, xq + (size_t)n * c.d,
                                     at<float>(ws, L.xq_s), s));
        if (c.n_shared)
            MOE_LAUNCH(launch_split_e4m3(c.T, c.d, x, c.T, nullptr, nullptr, xsq, xsq + (size_t)c.T * c.d,
                                         at<float>(ws, L.xsq_s), s));
    }
    {
        StageScope scope(kStageUp, s);
        if (use_decode_gemm(c)) {
            // split-K: the CTA that writes a tile's last K slice applies the SwiGLU itself
            MOE_LAUNCH(launch_gemm_decode(kGemmSwiGLU, up, np, status, sms, s, sp.up, w8 != nullptr,
                                          decode_tile_rows(c, w8 != nullptr), sp.up_balanced,
                                          sp.up > 1 ? at<unsigned int>(ws, L.up_sync) : nullptr));
        } else if (w8) {
            MOE_LAUNCH(launch_gemm_tc_w8(kGemmSwiGLU, up, np, status, sms, s, sp.up));
            if (sp.up > 1) {
                MOE_LAUNCH(launch_swiglu_finalize(n, offsets + c.E, c.d_ff, sp.up, up[0].part, h, nullptr, s));
                if (c.n_shared)
                    MOE_LAUNCH(launch_swiglu_finalize(c.T, nullptr, c.d_ff_shared, sp.up, up[1].part, hs, nullptr, s));
            }
        } else if (c.dtype == MOE_BF16) {
            MOE_LAUNCH(launch_gemm_tc(kGemmSwiGLU, up, np, status, sms, s, sp.up,
                                      use_pair_gemm(c) && sp.up == 1 && !up[0].a_gather));
            if (sp.up > 1) {
                MOE_LAUNCH(launch_swiglu_finalize(n, offsets + c.E, c.d_ff, sp.up, up[0].part, h, h_lo, s));
                if (c.n_shared)
                    MOE_LAUNCH(launch_swiglu_finalize(c.T, nullptr, c.d_ff_shared, sp.up, up[1].part, hs, hs_lo, s));
            }
        } else {
            MOE_LAUNCH(launch_gemm_simt_f32(kGemmSwiGLU, up, np, s));
        }
    }
    {
        StageScope scope(kStageDown, s);
        if (use_decode_gemm(c)) {
            if (q8) {
                MOE_LAUNCH(launch_split_e4m3(n, c.d_ff, h, n, nullptr, offsets + c.E, hq, hq + (size_t)n * c.d_ff,
                                             at<float>(ws, L.hq_s), s));
                if (c.n_shared)
                    MOE_LAUNCH(launch_split_e4m3(c.T, c.d_ff_shared, hs, c.T, nullptr, nullptr, hsq,
                                                 hsq + (size_t)c.T * c.d_ff_shared, at<float>(ws, L.hsq_s), s));
            }
            MOE_LAUNCH(launch_gemm_decode(kGemmScale, down, np, status, sms, s, sp.down, w8 != nullptr,
                                          decode_tile_rows(c, w8 != nullptr)));
            if (sp.down > 1 && reduce_down) {
                MOE_LAUNCH(launch_reduce_partials(n, offsets + c.E, c.d, sp.down, down[0].part, y_perm, s, c.yperm_bf16 != 0));
                if (c.n_shared)
                    MOE_LAUNCH(launch_reduce_partials(c.T, nullptr, c.d, sp.down, down[1].part, y_shared, s, c.yperm_bf16 != 0));
            }
        } else if (w8) {
            MOE_LAUNCH(launch_gemm_tc_w8(kGemmScale, down, np, status, sms, s, sp.down));
            if (sp.down > 1 && reduce_down) {
                MOE_LAUNCH(launch_reduce_partials(n, offsets + c.E, c.d, sp.down, down[0].part, y_perm, s, c.yperm_bf16 != 0));
                if (c.n_shared)
                    MOE_LAUNCH(launch_reduce_partials(c.T, nullptr, c.d, sp.down, down[1].part, y_shared, s, c.yperm_bf16 != 0));
            }
        } else if (c.dtype == MOE_BF16) {
            MOE_LAUNCH(launch_gemm_tc(split ? kGemmScaleSplit : kGemmScale, down, np, status, sms, s, sp.down,
                                      use_pair_gemm(c) && sp.down == 1));
            if (sp.down > 1 && reduce_down) {
                MOE_LAUNCH(launch_reduce_partials(n, offsets + c.E, c.d, sp.down, down[0].part, y_perm, s, c.yperm_bf16 != 0));
                if (c.n_shared)
                    MOE_LAUNCH(launch_reduce_partials(c.T, nullptr, c.d, sp.down, down[1].part, y_shared, s, c.yperm_bf16 != 0));
            }
        } else {
            MOE_LAUNCH(launch_gemm_simt_f32(kGemmScale, down, np, s));
        }
    }
    return MOE_OK;
}

// Expert-FFN rows in place (explicit gather, or the up GEMM's own gather
// for decode-sized batches), both GEMMs, combine over `slots` slots per
// token -- the part of moe_forward shared by both routings.
int forward_tail(const moe_config& c, const Layout& L, void* ws, const void* x, const int32_t* offsets,
                 const int32_t* sorted, const float* gates_perm, const int32_t* slot_pos, int slots, const void* w1,
                 const void* w3, const void* w2, const void* ws1, const void* ws3, const void* ws2, void* y,
                 int32_t* n_empty, int sms, cudaStream_t s, const moe_fp8_weights* w8) {
    int* status = at<int>(ws, L.status);
    void* x_perm = nullptr;
    const int32_t* gather_idx = nullptr;
    // FP8 decode batches: the E4M3 split of x puts the rows in expert order itself
    if (use_gather_a(c) || (w8 && use_decode_gemm(c))) {
        gather_idx = sorted;
    } else {
        x_perm = at<void>(ws, L.x_perm);
        StageScope scope(kStageGather, s);
        MOE_LAUNCH(launch_gather_rows(c.dtype, c.T, c.d, (int)perm_rows(c), offsets + c.E, sorted, x, x_perm,
                                      status, s));
    }
    void* y_perm = at<void>(ws, L.y_perm);
    void* y_shared = c.n_shared ? at<void>(ws, L.y_shared) : nullptr;
    MOE_TRY(enqueue_ffn(c, L, ws, x_perm, offsets, gates_perm, w1, w3, w2, x, ws1, ws3, ws2, y_perm, y_shared, sms,
                        s, false, gather_idx, w8));
    // combine (straight from the down GEMM's split-K slices when it was split;
    // a layer that keeps its expert rows in bf16 rounds each entry's slice sum
    // as the reduction into a bf16 row would)
    const Splits sp = choose_splits(c, w8 != nullptr);
    const int ydt = c.y_fp32 ? MOE_F32 : c.dtype;
    StageScope scope(kStageCombine, s);
    if (sp.down > 1) {
        MOE_LAUNCH(launch_combine_split(ydt, c.T, c.d, slots, at<float>(ws, L.part_dn), (size_t)perm_rows(c) * c.d,
                                        sp.down, slot_pos, c.n_shared ? at<float>(ws, L.part_dn_shared) : nullptr,
                                        (size_t)c.T * c.d, sp.down, y, s, n_empty, c.yperm_bf16 != 0));
    } else {
        MOE_LAUNCH(launch_combine(ydt, c.T, c.d, slots, y_perm, slot_pos, y_shared, y, s, n_empty, c.yperm_bf16 != 0));
    }
    return MOE_OK;
}

int forward_expert_choice(const moe_config& c, const Layout& L, void* ws, const void* x, const void* w_gate,
                          const float* logit_bias, const void* w1, const void* w3, const void* w2, const void* ws1,
                          const void* ws3, const void* ws2, void* y, const moe_stats* stats, int nblk, int sms,
                          cudaStream_t s, const moe_fp8_weights* w8) {
    const int C = ec_bucket(c);
    float* probs = at<float>(ws, L.probs);
    int32_t* sorted = at<int32_t>(ws, L.sorted);
    float* gates_perm = at<float>(ws, L.gates_perm);
    int32_t* slot_pos = at<int32_t>(ws, L.slot_pos);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* counts = (stats && stats->counts) ? stats->counts : at<int32_t>(ws, L.counts);
    int32_t* kept = (stats && stats->kept) ? stats->kept : at<int32_t>(ws, L.kept);
    int32_t* n_empty = stats ? stats->n_dropped : nullptr;
    MOE_TRY(enqueue_route_ec(c, L, ws, x, w_gate, logit_bias, probs, sorted, gates_perm, slot_pos, counts, kept,
                             offsets, n_empty, sms, s));
    if (stats && (stats->f || stats->p || stats->L)) {
        float* p_mean = stats->p ? stats->p : at<float>(ws, L.p_mean);
        StageScope scope(kStageScan, s);
        MOE_LAUNCH(launch_p_mean(c.T, c.E, nblk, at<float>(ws, L.p_part), p_mean, s));
        // f = counts / (E C): the E*C chosen pairs are the decisions
        if (stats->f || stats->L)
            MOE_LAUNCH(launch_load_stats(c.E * C, c.E, 1, c.alpha, counts, p_mean, stats->f, stats->L, s));
    }
    return forward_tail(c, L, ws, x, offsets, sorted, gates_perm, slot_pos, c.E, w1, w3, w2, ws1, ws3, ws2, y,
                        n_empty, sms, s, w8);
}

}  // namespace

bool test_stall_gemm() { return g_test_stall.load(std::memory_order_relaxed) != 0; }

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(const moe_config* cfg) {
    if (check_config(cfg) != MOE_OK) return 0;
    return layout(*cfg).total;
}

int moe_workspace_init(const moe_config* cfg, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    const Layout L = layout(*cfg);
    MOE_CUDA(cudaMemsetAsync(at<int>(ws, L.status), 0, 16, reinterpret_cast<cudaStream_t>(stream)));
    if (L.up_sync_bytes)
        MOE_CUDA(cudaMemsetAsync(at<int>(ws, L.up_sync), 0, L.up_sync_bytes, reinterpret_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

int moe_route(const moe_config* cfg, const void* x, const void* w_gate, const float* logit_bias,
              const float* select_bias, int32_t* topk_ids, float* gates, float* p_mean, void* ws, size_t ws_bytes,
              moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    if (expert_choice(*cfg)) return MOE_ERR_SHAPE;  // token-choice step
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!x || !w_gate || !topk_ids || !gates) return MOE_ERR_NULL;
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    for (const void* p : {x, w_gate, (const void*)topk_ids, (const void*)gates})
        if (!aligned16(p)) return MOE_ERR_ALIGN;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Layout L = layout(c);
    MOE_TRY(enqueue_route(c, L, ws, x, w_gate, logit_bias, select_bias, topk_ids, gates, nullptr, sms, s, c.k));
    if (p_mean) {
        const int ch = router_chunk(c.T, c.E, c.d, c.dtype);
        const int nblk = (c.T + ch - 1) / ch;
        StageScope scope(kStageRouter, s);
        MOE_LAUNCH(launch_p_mean(c.T, c.E, nblk, at<float>(ws, L.p_part), p_mean, s));
    }
    return MOE_OK;
}

int moe_route_expert_choice(const moe_config* cfg, const void* x, const void* w_gate, const float* logit_bias,
                            float* probs, int32_t* sorted_token_ids, float* gates_perm, int32_t* slot_pos,
                            int32_t* offsets, float* p_mean, void* x_perm, void* ws, size_t ws_bytes,
                            moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    const moe_config& c = *cfg;
    if (!expert_choice(c)) return MOE_ERR_SHAPE;
    if (c.T == 0) return MOE_OK;
    if (!x || !w_gate || !sorted_token_ids || !gates_perm || !slot_pos || !offsets) return MOE_ERR_NULL;
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    if (!aligned16(x) || !aligned16(w_gate) || (x_perm && !aligned16(x_perm))) return MOE_ERR_ALIGN;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Layout L = layout(c);
    float* pr = probs ? probs : at<float>(ws, L.probs);
    MOE_TRY(enqueue_route_ec(c, L, ws, x, w_gate, logit_bias, pr, sorted_token_ids, gates_perm, slot_pos, nullptr,
                             nullptr, offsets, nullptr, sms, s));
    if (p_mean) {
        const int ch = router_chunk(c.T, c.E, c.d, c.dtype);
        StageScope scope(kStageRouter, s);
        MOE_LAUNCH(launch_p_mean(c.T, c.E, (c.T + ch - 1) / ch, at<float>(ws, L.p_part), p_mean, s));
    }
    if (x_perm) {
        StageScope scope(kStageGather, s);
        MOE_LAUNCH(launch_gather_rows(c.dtype, c.T, c.d, (int)perm_rows(c), offsets + c.E, sorted_token_ids, x,
                                      x_perm, at<int>(ws, L.status), s));
    }
    return MOE_OK;
}

int moe_permute(const moe_config* cfg, const int32_t* topk_ids, const float* gates, const void* x, int32_t* counts,
                int32_t* kept, int32_t* offsets, int32_t* sorted_token_ids, int32_t* slot_pos, float* gates_perm,
                void* x_perm, int32_t* n_dropped, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    if (expert_choice(*cfg)) return MOE_ERR_SHAPE;  // token-choice step
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!topk_ids || !gates || !x || !counts || !kept || !offsets || !sorted_token_ids || !slot_pos ||
        !gates_perm || !x_perm || !n_dropped)
        return MOE_ERR_NULL;
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_ALIGN;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Layout L = layout(c);
    int* status = at<int>(ws, L.status);
    int32_t* block_hist = at<int32_t>(ws, L.block_hist);
    GroupOut o{};
    o.counts = counts;
    o.kept = kept;
    o.offsets = offsets;
    o.sorted_token_ids = sorted_token_ids;
    o.slot_pos = slot_pos;
    o.gates_perm = gates_perm;
    o.n_dropped = n_dropped;
    {
        StageScope scope(kStageScan, s);
        const int chunk = kRouterTokensPerBlock;
        MOE_LAUNCH(launch_group_hist(c.T, c.E, c.k, chunk, topk_ids, block_hist, status, s));
        MOE_LAUNCH(launch_group_scan(c.T, c.E, c.k, chunk, c.capacity, topk_ids, gates, block_hist, o, status, s));
    }
    StageScope scope(kStageGather, s);
    MOE_LAUNCH(launch_gather_rows(c.dtype, c.T, c.d, c.T * c.k, offsets + c.E, sorted_token_ids, x, x_perm, status, s));
    return MOE_OK;
}

int moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets, const float* gates_perm,
                   const void* w1, const void* w3, const void* w2, const void* x, const void* ws1, const void* ws3,
                   const void* ws2, void* y_perm, void* y_shared, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!x_perm || !offsets || !gates_perm || !w1 || !w3 || !w2 || !y_perm) return MOE_ERR_NULL;
    if (c.n_shared && (!x || !ws1 || !ws3 || !ws2 || !y_shared)) return MOE_ERR_NULL;
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    for (const void* p : {x_perm, w1, w3, w2, (const void*)y_perm})
        if (!aligned16(p)) return MOE_ERR_ALIGN;
    if (c.n_shared)
        for (const void* p : {x, ws1, ws3, ws2, (const void*)y_shared})
            if (!aligned16(p)) return MOE_ERR_ALIGN;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    const Layout L = layout(c);
    return enqueue_ffn(c, L, ws, x_perm, offsets, gates_perm, w1, w3, w2, x, ws1, ws3, ws2, y_perm, y_shared, sms,
                       reinterpret_cast<cudaStream_t>(stream), true, nullptr);
}

int moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* slot_pos, const void* y_shared, void* y,
                moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!y_perm || !slot_pos || !y) return MOE_ERR_NULL;
    if (!aligned16(y_perm) || !aligned16(y) || (y_shared && !aligned16(y_shared))) return MOE_ERR_ALIGN;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    StageScope scope(kStageCombine, reinterpret_cast<cudaStream_t>(stream));
    MOE_LAUNCH(launch_combine(c.y_fp32 ? MOE_F32 : c.dtype, c.T, c.d, slots_per_token(c), y_perm, slot_pos, y_shared, y,
                              reinterpret_cast<cudaStream_t>(stream), nullptr, c.yperm_bf16 != 0));
    return MOE_OK;
}

int moe_load_stats(const moe_config* cfg, const int32_t* counts, const float* p_mean, float* f, float* L,
                   moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!counts || !p_mean) return MOE_ERR_NULL;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    // decisions: T k, or the E C chosen pairs under expert choice
    const int tn = expert_choice(c) ? (int)perm_rows(c) : c.T, kk = expert_choice(c) ? 1 : c.k;
    MOE_LAUNCH(launch_load_stats(tn, c.E, kk, c.alpha, counts, p_mean, f, L, reinterpret_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

int moe_bias_update(const moe_config* cfg, const int32_t* counts, float gamma, float* select_bias,
                    moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    if (expert_choice(*cfg)) return MOE_ERR_SHAPE;  // token-choice step
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!counts || !select_bias) return MOE_ERR_NULL;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    MOE_LAUNCH(launch_bias_update(c.T, c.E, c.k, counts, gamma, select_bias, reinterpret_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

// Steps 1-7 for batches the two fused decode kernels take (decode_fused.cu):
// every CTA routes the batch itself, so the router, the grouping, the x gather
// and the combine have no launch of their own.  H goes through the workspace.
static int forward_fused_decode(const moe_config& c, const FusedPlan& fp, const Layout& L, void* ws, const void* x,
                                const void* w_gate, const float* logit_bias, const float* select_bias,
                                const void* w1, const void* w3, const void* w2, const void* ws1, const void* ws3,
                                const void* ws2, const moe_fp8_weights* w8, void* y, const moe_stats* stats,
                                cudaStream_t s) {
    FusedDecodeArgs a{};
    a.T = c.T;
    a.d = c.d;
    a.E = c.E;
    a.k = c.k;
    a.F = c.d_ff;
    a.Fs = c.n_shared ? c.d_ff_shared : 0;
    a.n_shared = c.n_shared;
    a.renormalize = c.renormalize;
    a.capacity = c.capacity;
    a.y_fp32 = c.y_fp32;
    a.fp8 = w8 != nullptr;
    a.alpha = c.alpha;
    a.x = x;
    a.wg = w_gate;
    a.logit_bias = logit_bias;
    a.select_bias = select_bias;
    a.w1 = w1;
    a.w3 = w3;
    a.w2 = w2;
    a.ws1 = ws1;
    a.ws3 = ws3;
    a.ws2 = ws2;
    if (w8) {
        a.s1 = w8->s1;
        a.s3 = w8->s3;
        a.s2 = w8->s2;
        a.ss1 = w8->ss1;
        a.ss3 = w8->ss3;
        a.ss2 = w8->ss2;
    }
    a.h = at<void>(ws, L.h);
    a.h_shared = c.n_shared ? at<void>(ws, L.h_shared) : nullptr;
    a.y = y;
    if (stats) {
        a.counts = stats->counts;
        a.kept = stats->kept;
        a.n_dropped = stats->n_dropped;
        a.f = stats->f;
        a.p = stats->p;
        a.L = stats->L;
    }
    a.status = at<int>(ws, L.status);
    {
        StageScope scope(kStageUp, s);
        MOE_LAUNCH(launch_fused_up(a, fp, s));
    }
    StageScope scope(kStageDown, s);
    MOE_LAUNCH(launch_fused_down(a, fp, s));
    return MOE_OK;
}

// Steps 1-7 after argument checks; w8 != nullptr: FP8 expert weights.
static int forward_body(const moe_config& c, const void* x, const void* w_gate, const float* logit_bias,
                        const float* select_bias, const void* w1, const void* w3, const void* w2, const void* ws1,
                        const void* ws3, const void* ws2, const moe_fp8_weights* w8, void* y, const moe_stats* stats,
                        void* ws, cudaStream_t s, int sms) {
    const Layout L = layout(c);
    int* status = at<int>(ws, L.status);
    int32_t* topk_ids = at<int32_t>(ws, L.topk_ids);
    float* gates = at<float>(ws, L.gates);
    int32_t* block_hist = at<int32_t>(ws, L.block_hist);
    const int chunk = router_chunk(c.T, c.E, c.d, c.dtype);
    const int nblk = (c.T + chunk - 1) / chunk;
    if (expert_choice(c))
        return forward_expert_choice(c, L, ws, x, w_gate, logit_bias, w1, w3, w2, ws1, ws3, ws2, y, stats, nblk,
                                     sms, s, w8);
    const FusedPlan fp = fused_decode_plan(c, w8 != nullptr, sms);
    if (fp.ok)
        return forward_fused_decode(c, fp, L, ws, x, w_gate, logit_bias, select_bias, w1, w3, w2, ws1, ws3, ws2, w8,
                                    y, stats, s);

    // 1-4: router, softmax, top-k (the router blocks also emit their id
    // histograms), grouping (+ load statistics from the router's partial sums)
    GroupOut o{};
    o.counts = (stats && stats->counts) ? stats->counts : at<int32_t>(ws, L.counts);
    o.kept = (stats && stats->kept) ? stats->kept : at<int32_t>(ws, L.kept);
    o.offsets = at<int32_t>(ws, L.offsets);
    o.sorted_token_ids = at<int32_t>(ws, L.sorted);
    o.slot_pos = at<int32_t>(ws, L.slot_pos);
    o.gates_perm = at<float>(ws, L.gates_perm);
    o.n_dropped = (stats && stats->n_dropped) ? stats->n_dropped : at<int32_t>(ws, L.n_dropped);
    if (stats && (stats->f || stats->p || stats->L)) {
        o.p_part = at<float>(ws, L.p_part);
        o.p_nblk = nblk;
        o.f = stats->f;
        o.p_mean = stats->p;
        o.L = stats->L;
        o.alpha = c.alpha;
    }
    MOE_TRY(enqueue_route_group(c, L, ws, x, w_gate, logit_bias, select_bias, topk_ids, gates, o, sms, s));
    // 5-6: rows in expert order (decode-sized bf16 batches: the up GEMM
    // gathers x rows itself with TMA gather4), expert FFNs (routed groups +
    // shared expert in the same launches), combine
    return forward_tail(c, L, ws, x, o.offsets, o.sorted_token_ids, o.gates_perm, o.slot_pos, c.k, w1, w3, w2, ws1,
                        ws3, ws2, y, nullptr, sms, s, w8);
}

int moe_forward(const moe_config* cfg, const void* x, const void* w_gate, const float* logit_bias,
                const float* select_bias, const void* w1, const void* w3, const void* w2, const void* ws1,
                const void* ws3, const void* ws2, void* y, const moe_stats* stats, void* ws, size_t ws_bytes,
                moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    const moe_config& c = *cfg;
    if (c.T == 0) return MOE_OK;
    if (!x || !w_gate || !w1 || !w3 || !w2 || !y) return MOE_ERR_NULL;
    if (c.n_shared && (!ws1 || !ws3 || !ws2)) return MOE_ERR_NULL;
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    for (const void* p : {x, w_gate, w1, w3, w2, (const void*)y})
        if (!aligned16(p)) return MOE_ERR_ALIGN;
    if (c.n_shared)
        for (const void* p : {ws1, ws3, ws2})
            if (!aligned16(p)) return MOE_ERR_ALIGN;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    return forward_body(c, x, w_gate, logit_bias, select_bias, w1, w3, w2, ws1, ws3, ws2, nullptr, y, stats, ws,
                        reinterpret_cast<cudaStream_t>(stream), sms);
}

int moe_forward_fp8(const moe_config* cfg, const void* x, const void* w_gate, const float* logit_bias,
                    const float* select_bias, const moe_fp8_weights* w, void* y, const moe_stats* stats, void* ws,
                    size_t ws_bytes, moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    const moe_config& c = *cfg;
    if (c.dtype != MOE_BF16 || c.h_split != 0) return MOE_ERR_DTYPE;
    if (c.d % 16 || c.d_ff % 16 || (c.n_shared && c.d_ff_shared % 16)) return MOE_ERR_SHAPE;
    if (c.T == 0) return MOE_OK;
    if (!w || !x || !w_gate || !y || !w->w1 || !w->w3 || !w->w2 || !w->s1 || !w->s3 || !w->s2) return MOE_ERR_NULL;
    if (c.n_shared && (!w->ws1 || !w->ws3 || !w->ws2 || !w->ss1 || !w->ss3 || !w->ss2)) return MOE_ERR_NULL;
    MOE_TRY(check_ws(cfg, ws, ws_bytes));
    for (const void* p : {x, w_gate, (const void*)y, (const void*)w->w1, (const void*)w->w3, (const void*)w->w2,
                          (const void*)w->s1, (const void*)w->s3, (const void*)w->s2})
        if (!aligned16(p)) return MOE_ERR_ALIGN;
    if (c.n_shared)
        for (const void* p : {(const void*)w->ws1, (const void*)w->ws3, (const void*)w->ws2, (const void*)w->ss1,
                              (const void*)w->ss3, (const void*)w->ss2})
            if (!aligned16(p)) return MOE_ERR_ALIGN;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    return forward_body(c, x, w_gate, logit_bias, select_bias, w->w1, w->w3, w->w2, w->ws1, w->ws3, w->ws2, w, y,
                        stats, ws, reinterpret_cast<cudaStream_t>(stream), sms);
}

int moe_quantize_fp8(const void* w, int32_t dtype, int64_t rows, int32_t cols, uint8_t* q, float* scale,
                     moe_stream_t stream) {
    if (dtype != MOE_BF16 && dtype != MOE_F32) return MOE_ERR_DTYPE;
    if (rows < 0 || cols < 16 || cols % 16) return MOE_ERR_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!w || !q || !scale) return MOE_ERR_NULL;
    if (!aligned16(w) || !aligned16(q) || !aligned16(scale)) return MOE_ERR_ALIGN;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    MOE_LAUNCH(launch_quantize_fp8(dtype, rows, cols, w, q, scale, reinterpret_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

size_t moe_backward_workspace_size(const moe_config* cfg) {
    if (check_config(cfg) != MOE_OK || cfg->dtype != MOE_BF16 || expert_choice(*cfg)) return 0;
    return blayout(*cfg).total;
}

// moe_backward and moe_backward_saved: saved = the routing, grouping, x rows
// in expert order, softmax rows and G, U of the layer call are the ones
// moe_forward_train left in ws, so they are not recomputed.
static int backward_impl(const moe_config* cfg, const void* x, const void* w_gate, const float* logit_bias,
                         const float* select_bias, const void* w1, const void* w3, const void* w2, const void* ws1,
                         const void* ws3, const void* ws2, const void* dy, float dL, float* dx, float* dw_gate,
                         float* dw1, float* dw3, float* dw2, float* dws1, float* dws3, float* dws2, void* ws,
                         size_t ws_bytes, moe_stream_t stream, bool saved) {
    MOE_TRY(check_config(cfg));
    const moe_config& c = *cfg;
    if (c.dtype != MOE_BF16) return MOE_ERR_DTYPE;
    if (expert_choice(c)) return MOE_ERR_SHAPE;  // token choice only
    if (c.T == 0) return MOE_OK;
    if (!x || !w_gate || !w1 || !w3 || !w2 || !dy || !dx || !dw_gate || !dw1 || !dw3 || !dw2 || !ws)
        return MOE_ERR_NULL;
    if (c.n_shared && (!ws1 || !ws3 || !ws2 || !dws1 || !dws3 || !dws2)) return MOE_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(ws) % kAlign) return MOE_ERR_WORKSPACE;
    const BLayout B = blayout(c);
    if (ws_bytes < B.total) return MOE_ERR_WORKSPACE;
    for (const void* p : {x, w_gate, w1, w3, w2, dy, (const void*)dx, (const void*)dw_gate, (const void*)dw1,
                          (const void*)dw3, (const void*)dw2})
        if (!aligned16(p)) return MOE_ERR_ALIGN;
    if (c.n_shared)
        for (const void* p : {ws1, ws3, ws2, (const void*)dws1, (const void*)dws3, (const void*)dws2})
            if (!aligned16(p)) return MOE_ERR_ALIGN;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Layout L = layout(c);
    const int E = c.E, F = c.d_ff, d = c.d, T = c.T, Fs = c.d_ff_shared, n = c.T * c.k;
    int* status = at<int>(ws, L.status);
    int32_t* topk_ids = at<int32_t>(ws, L.topk_ids);
    float* gates = at<float>(ws, L.gates);
    float* probs = at<float>(ws, B.probs);
    const int chunk = router_chunk(c.T, c.E, c.d, c.dtype);

    // forward routing and grouping again (the decisions the gradients hold fixed)
    GroupOut o{};
    o.counts = at<int32_t>(ws, L.counts);
    o.kept = at<int32_t>(ws, L.kept);
    o.offsets = at<int32_t>(ws, L.offsets);
    o.sorted_token_ids = at<int32_t>(ws, L.sorted);
    o.slot_pos = at<int32_t>(ws, L.slot_pos);
    o.gates_perm = at<float>(ws, L.gates_perm);
    o.n_dropped = at<int32_t>(ws, L.n_dropped);
    if (!saved)
        MOE_TRY(enqueue_route_group(c, L, ws, x, w_gate, logit_bias, select_bias, topk_ids, gates, o, sms, s, probs));
    const int32_t* rows_end = o.offsets + E;
    void* xp = at<void>(ws, B.xp);
    void* dyp = at<void>(ws, B.dyp);
    if (!saved) MOE_LAUNCH(launch_gather_rows(MOE_BF16, T, d, n, rows_end, o.sorted_token_ids, x, xp, status, s));
    MOE_LAUNCH(launch_gather_rows(MOE_BF16, T, d, n, rows_end, o.sorted_token_ids, dy, dyp, status, s));
    int32_t* kbase = at<int32_t>(ws, B.kbase);
    int32_t* klen = at<int32_t>(ws, B.klen);
    MOE_LAUNCH(launch_k_windows(E, o.offsets, kbase, klen, -1, s));
    int32_t *s_off = nullptr, *s_kbase = nullptr, *s_klen = nullptr;
    if (c.n_shared) {
        s_off = at<int32_t>(ws, B.s_off);
        s_kbase = at<int32_t>(ws, B.s_kbase);
        s_klen = at<int32_t>(ws, B.s_klen);
        MOE_LAUNCH(launch_k_windows(1, s_off, s_kbase, s_klen, T, s));
    }

    // grouped GEMMs of the routed experts (problem 0) and the shared expert (problem 1)
    const int np = c.n_shared ? 2 : 1;
    auto routed = [&](const void* A, int a_rows, const void* Bm, int N, int K, void* out) {
        GemmProblem g{};
        g.A = A;
        g.a_rows = a_rows;
        g.B1 = Bm;
        g.offsets = o.offsets;
        g.G = E;
        g.N = N;
        g.K = K;
        g.out = out;
        return g;
    };
    auto dense = [&](const void* A, int M, const void* Bm, int N, int K, void* out) {
        GemmProblem g{};
        g.A = A;
        g.a_rows = M;
        g.B1 = Bm;
        g.G = 1;
        g.M = M;
        g.N = N;
        g.K = K;
        g.out = out;
        return g;
    };
    // products with W^T read the weights as they are stored: MN-major B
    auto transposed = [&](GemmProblem g, const void* b2, int kpart) {
        g.b_mn = 1;
        g.B2 = b2;
        g.kpart = kpart;
        return g;
    };
    auto windows = [&](const void* A, int M, const void* Bm, int N, int K, const int32_t* kb, const int32_t* kl, int G,
                       void* out) {
        GemmProblem g{};
        g.A = A;
        g.a_rows = M;
        g.B1 = Bm;
        g.G = G;
        g.M = M;
        g.N = N;
        g.K = K;
        g.kbase = kb;
        g.klen = kl;
        g.out = out;
        return g;
    };
    float* G = at<float>(ws, B.G);
    float* U = at<float>(ws, B.U);
    float* D = at<float>(ws, B.D);
    // large segments: every product runs on CTA pairs (Scale mode without
    // gates is the plain product)
    const bool pair = use_pair_gemm(c);
    const int pm = pair ? kGemmScale : kGemmPlain;
    if (!saved) {
        GemmProblem p1[2] = {routed(xp, n, w1, F, d, G), dense(x, T, ws1, Fs, d, at<float>(ws, B.Gs))};
        MOE_LAUNCH(launch_gemm_tc(pm, p1, np, status, sms, s, 1, pair));
        GemmProblem p2[2] = {routed(xp, n, w3, F, d, U), dense(x, T, ws3, Fs, d, at<float>(ws, B.Us))};
        MOE_LAUNCH(launch_gemm_tc(pm, p2, np, status, sms, s, 1, pair));
    }
    // D = dy W2 (W2 stored [d][F]: B^T of this product), consumed in the GEMM's
    // epilogue by the SwiGLU backward: dGU = [dG | dU], Hb = bf16(h), and the
    // gate gradients dg = sum_f D h as one partial per 256-column tile (the D
    // region holds them), summed in tile order below
    void* dGU = at<void>(ws, B.dGU);
    void* Hb = at<void>(ws, B.Hb);
    float* dgp = at<float>(ws, B.dgp);
    const int dg_ld = (n + 3) / 4 * 4;
    const int dg_tiles = (F + 255) / 256;
    {
        GemmProblem p3[2] = {transposed(routed(dyp, n, w2, F, d, nullptr), nullptr, 0),
                             transposed(dense(dy, T, ws2, Fs, d, nullptr), nullptr, 0)};
        p3[0].row_scale = o.gates_perm;
        p3[0].bwd_G = G;
        p3[0].bwd_U = U;
        p3[0].bwd_dGU = dGU;
        p3[0].bwd_Hb = Hb;
        p3[0].bwd_dgp_part = D;
        p3[0].bwd_dgp_ld = dg_ld;
        p3[1].bwd_G = at<float>(ws, B.Gs);
        p3[1].bwd_U = at<float>(ws, B.Us);
        p3[1].bwd_dGU = at<void>(ws, B.dGUs);
        p3[1].bwd_Hb = at<void>(ws, B.Hbs);
        MOE_LAUNCH(launch_gemm_tc(kGemmSwigluBwd, p3, np, status, sms, s, 1, pair));
        MOE_LAUNCH(launch_reduce_partials(1, nullptr, dg_ld, dg_tiles, D, dgp, s));
    }
    float* dXp = at<float>(ws, B.dXp);
    float* dXs = c.n_shared ? at<float>(ws, B.dXs) : nullptr;
    {
        // dX = dG W1 + dU W3: K in two parts (dG with W1, dU with W3), W1 and W3 stored [F][d]
        GemmProblem p4[2] = {transposed(routed(dGU, n, w1, d, 2 * F, dXp), w3, F),
                             transposed(dense(at<void>(ws, B.dGUs), T, ws1, d, 2 * Fs, dXs), ws3, Fs)};
        MOE_LAUNCH(launch_gemm_tc(pm, p4, np, status, sms, s, 1, pair));
    }

    // weight gradients: per-expert K windows of the transposed activations
    const int nc = B.ncols, ncs = B.ncols_s;
    void* dGT = at<void>(ws, B.dGT);
    void* dUT = at<void>(ws, B.dUT);
    void* HbT = at<void>(ws, B.HbT);
    void* xpT = at<void>(ws, B.xpT);
    void* dysT = at<void>(ws, B.dysT);
    // the dG|dU rows in one pass: source column c < F lands in dG^T's row c, c >= F in dU^T's row c - F
    MOE_LAUNCH(launch_transpose_windows(dGU, 2 * (size_t)F, 0, 2 * F, E, o.offsets, kbase, klen, nullptr, dGT, nc, nc,
                                        s));
    MOE_LAUNCH(launch_transpose_windows(Hb, F, 0, F, E, o.offsets, kbase, klen, nullptr, HbT, nc, nc, s));
    MOE_LAUNCH(launch_transpose_windows(xp, d, 0, d, E, o.offsets, kbase, klen, nullptr, xpT, nc, nc, s));
    MOE_LAUNCH(launch_transpose_windows(dyp, d, 0, d, E, o.offsets, kbase, klen, o.gates_perm, dysT, nc, nc, s));
    if (c.n_shared) {
        void* dGUs = at<void>(ws, B.dGUs);
        MOE_LAUNCH(launch_transpose_windows(dGUs, 2 * (size_t)Fs, 0, 2 * Fs, 1, s_off, s_kbase, s_klen, nullptr,
                                            at<void>(ws, B.dGsT), ncs, ncs, s));
        MOE_LAUNCH(launch_transpose_windows(at<void>(ws, B.Hbs), Fs, 0, Fs, 1, s_off, s_kbase, s_klen, nullptr,
                                            at<void>(ws, B.HbsT), ncs, ncs, s));
        MOE_LAUNCH(launch_transpose_windows(x, d, 0, d, 1, s_off, s_kbase, s_klen, nullptr, at<void>(ws, B.xT), ncs,
                                            ncs, s));
        MOE_LAUNCH(launch_transpose_windows(dy, d, 0, d, 1, s_off, s_kbase, s_klen, nullptr, at<void>(ws, B.dyT), ncs,
                                            ncs, s));
    }
    {
        GemmProblem q1[2] = {windows(dGT, F, xpT, d, nc, kbase, klen, E, dw1),
                             windows(at<void>(ws, B.dGsT), Fs, at<void>(ws, B.xT), d, ncs, s_kbase, s_klen, 1, dws1)};
        MOE_LAUNCH(launch_gemm_tc(pm, q1, np, status, sms, s, 1, pair));
        GemmProblem q3[2] = {windows(dUT, F, xpT, d, nc, kbase, klen, E, dw3),
                             windows(at<void>(ws, B.dUsT), Fs, at<void>(ws, B.xT), d, ncs, s_kbase, s_klen, 1, dws3)};
        MOE_LAUNCH(launch_gemm_tc(pm, q3, np, status, sms, s, 1, pair));
        GemmProblem q2[2] = {windows(dysT, d, HbT, F, nc, kbase, klen, E, dw2),
                             windows(at<void>(ws, B.dyT), d, at<void>(ws, B.HbsT), Fs, ncs, s_kbase, s_klen, 1, dws2)};
        MOE_LAUNCH(launch_gemm_tc(pm, q2, np, status, sms, s, 1, pair));
    }

    // router: gate gradients -> logits (+ balance loss) -> W_g and x
    float* dlog = at<float>(ws, B.dlog);
    float* R = at<float>(ws, B.R);
    MOE_LAUNCH(launch_router_backward(T, E, c.k, probs, topk_ids, o.slot_pos, gates, dgp, c.renormalize, o.counts,
                                      c.alpha, dL, dlog, s));
    MOE_LAUNCH(launch_router_dx(MOE_BF16, T, E, d, dlog, w_gate, dXs, R, s));
    float* wgp = at<float>(ws, B.wg_part);
    const int wg_split = wgate_grad_split(E, d);
    MOE_LAUNCH(launch_wgate_grad(MOE_BF16, T, E, d, dlog, x, wg_split, wgp, s));
    MOE_LAUNCH(launch_reduce_partials(E, nullptr, d, wg_split, wgp, dw_gate, s));
    // dx = sum over kept slots of dX rows + router and shared-expert parts
    MOE_LAUNCH(launch_combine(MOE_F32, T, d, c.k, dXp, o.slot_pos, R, dx, s));
    return MOE_OK;
}

int moe_forward_train(const moe_config* cfg, const void* x, const void* w_gate, const float* logit_bias,
                      const float* select_bias, const void* w1, const void* w3, const void* w2, const void* ws1,
                      const void* ws3, const void* ws2, void* y, const moe_stats* stats, void* ws, size_t ws_bytes,
                      moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    const moe_config& c = *cfg;
    if (c.dtype != MOE_BF16) return MOE_ERR_DTYPE;
    if (expert_choice(c) || c.h_split) return MOE_ERR_SHAPE;  // token choice, single bf16 H
    if (c.T == 0) return MOE_OK;
    if (!x || !w_gate || !w1 || !w3 || !w2 || !y || !ws) return MOE_ERR_NULL;
    if (c.n_shared && (!ws1 || !ws3 || !ws2)) return MOE_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(ws) % kAlign) return MOE_ERR_WORKSPACE;
    const BLayout B = blayout(c);
    if (ws_bytes < B.total) return MOE_ERR_WORKSPACE;
    for (const void* p : {x, w_gate, w1, w3, w2, (const void*)y})
        if (!aligned16(p)) return MOE_ERR_ALIGN;
    if (c.n_shared)
        for (const void* p : {ws1, ws3, ws2})
            if (!aligned16(p)) return MOE_ERR_ALIGN;
    int sms = 0;
    MOE_TRY(device_sms(&sms));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const Layout L = layout(c);
    const int E = c.E, F = c.d_ff, d = c.d, T = c.T, Fs = c.d_ff_shared, n = c.T * c.k;
    int* status = at<int>(ws, L.status);
    int32_t* topk_ids = at<int32_t>(ws, L.topk_ids);
    float* gates = at<float>(ws, L.gates);
    const int chunk = router_chunk(c.T, c.E, c.d, c.dtype);
    const int nblk = (c.T + chunk - 1) / chunk;

    // 1-4: routing (softmax rows kept) and grouping, into the workspace regions
    // moe_backward_saved reads
    GroupOut o{};
    o.counts = at<int32_t>(ws, L.counts);
    o.kept = at<int32_t>(ws, L.kept);
    o.offsets = at<int32_t>(ws, L.offsets);
    o.sorted_token_ids = at<int32_t>(ws, L.sorted);
    o.slot_pos = at<int32_t>(ws, L.slot_pos);
    o.gates_perm = at<float>(ws, L.gates_perm);
    o.n_dropped = at<int32_t>(ws, L.n_dropped);
    if (stats && (stats->f || stats->p || stats->L)) {
        o.p_part = at<float>(ws, L.p_part);
        o.p_nblk = nblk;
        o.f = stats->f;
        o.p_mean = stats->p;
        o.L = stats->L;
        o.alpha = c.alpha;
    }
    MOE_TRY(enqueue_route_group(c, L, ws, x, w_gate, logit_bias, select_bias, topk_ids, gates, o, sms, s,
                                at<float>(ws, B.probs)));
    if (stats) {  // the counts stay in the workspace for the backward; copies for the caller
        if (stats->counts && cudaMemcpyAsync(stats->counts, o.counts, 4 * (size_t)E, cudaMemcpyDeviceToDevice, s))
            return MOE_ERR_CUDA;
        if (stats->kept && cudaMemcpyAsync(stats->kept, o.kept, 4 * (size_t)E, cudaMemcpyDeviceToDevice, s))
            return MOE_ERR_CUDA;
        if (stats->n_dropped && cudaMemcpyAsync(stats->n_dropped, o.n_dropped, 4, cudaMemcpyDeviceToDevice, s))
            return MOE_ERR_CUDA;
    }
    // 5: x rows in expert order
    void* xp = at<void>(ws, B.xp);
    MOE_LAUNCH(launch_gather_rows(MOE_BF16, T, d, n, o.offsets + E, o.sorted_token_ids, x, xp, status, s));
    // 6: expert FFNs; the up GEMM also keeps G and U (fp32) for the backward
    const bool pair = use_pair_gemm(c);
    const int np = c.n_shared ? 2 : 1;
    void* h = at<void>(ws, L.h);
    void* hs = at<void>(ws, L.h_shared);
    void* y_perm = at<void>(ws, L.y_perm);
    void* y_shared = c.n_shared ? at<void>(ws, L.y_shared) : nullptr;
    GemmProblem up[2] = {}, down[2] = {};
    up[0].A = xp;
    up[0].a_rows = n;
    up[0].B1 = w1;
    up[0].B2 = w3;
    up[0].offsets = o.offsets;
    up[0].G = E;
    up[0].N = F;
    up[0].K = d;
    up[0].out = h;
    up[0].out_g = at<float>(ws, B.G);
    up[0].out_u = at<float>(ws, B.U);
    down[0].A = h;
    down[0].a_rows = n;
    down[0].B1 = w2;
    down[0].offsets = o.offsets;
    down[0].G = E;
    down[0].N = d;
    down[0].K = F;
    down[0].out = y_perm;
    down[0].row_scale = o.gates_perm;
    if (c.n_shared) {
        up[1].A = x;
        up[1].a_rows = T;
        up[1].B1 = ws1;
        up[1].B2 = ws3;
        up[1].G = 1;
        up[1].M = T;
        up[1].N = Fs;
        up[1].K = d;
        up[1].out = hs;
        up[1].out_g = at<float>(ws, B.Gs);
        up[1].out_u = at<float>(ws, B.Us);
        down[1].A = hs;
        down[1].a_rows = T;
        down[1].B1 = ws2;
        down[1].G = 1;
        down[1].M = T;
        down[1].N = d;
        down[1].K = Fs;
        down[1].out = y_shared;
    }
    MOE_LAUNCH(launch_gemm_tc(kGemmSwiGLU, up, np, status, sms, s, 1, pair));
    MOE_LAUNCH(launch_gemm_tc(kGemmScale, down, np, status, sms, s, 1, pair));
    // 7: combine
    MOE_LAUNCH(launch_combine(c.y_fp32 ? MOE_F32 : c.dtype, T, d, c.k, y_perm, o.slot_pos, y_shared, y, s, nullptr,
                              c.yperm_bf16 != 0));
    return MOE_OK;
}

int moe_backward(const moe_config* cfg, const void* x, const void* w_gate, const float* logit_bias,
                 const float* select_bias, const void* w1, const void* w3, const void* w2, const void* ws1,
                 const void* ws3, const void* ws2, const void* dy, float dL, float* dx, float* dw_gate, float* dw1,
                 float* dw3, float* dw2, float* dws1, float* dws3, float* dws2, void* ws, size_t ws_bytes,
                 moe_stream_t stream) {
    return backward_impl(cfg, x, w_gate, logit_bias, select_bias, w1, w3, w2, ws1, ws3, ws2, dy, dL, dx, dw_gate, dw1,
                         dw3, dw2, dws1, dws3, dws2, ws, ws_bytes, stream, false);
}

int moe_backward_saved(const moe_config* cfg, const void* x, const void* w_gate, const float* logit_bias,
                       const float* select_bias, const void* w1, const void* w3, const void* w2, const void* ws1,
                       const void* ws3, const void* ws2, const void* dy, float dL, float* dx, float* dw_gate,
                       float* dw1, float* dw3, float* dw2, float* dws1, float* dws3, float* dws2, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
    return backward_impl(cfg, x, w_gate, logit_bias, select_bias, w1, w3, w2, ws1, ws3, ws2, dy, dL, dx, dw_gate, dw1,
                         dw3, dw2, dws1, dws3, dws2, ws, ws_bytes, stream, true);
}

int moe_last_device_status(const moe_config* cfg, void* ws, moe_stream_t stream) {
    MOE_TRY(check_config(cfg));
    if (!ws) return MOE_ERR_NULL;
    const Layout L = layout(*cfg);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(&v, at<int>(ws, L.status), sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (v != 0) {
        // a kernel that gave up may have left its counters mid-count: clear them with the word
        if (cudaMemset(at<int>(ws, L.status), 0, 16) != cudaSuccess) return MOE_ERR_CUDA;
        if (L.up_sync_bytes && cudaMemset(at<int>(ws, L.up_sync), 0, L.up_sync_bytes) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return v;
}

const char* moe_strerror(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_NULL: return "a required pointer is NULL";
        case MOE_ERR_SHAPE: return "sizes out of range or not multiples of 8";
        case MOE_ERR_DTYPE: return "unknown dtype";
        case MOE_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
        case MOE_ERR_CUDA: return "a CUDA launch or runtime call failed";
        case MOE_ERR_DEVICE: return "the current device is not a compute-capability 10.3 GPU";
        case MOE_ERR_TIMEOUT: return "a kernel's bounded wait ran out (device status)";
        case MOE_ERR_DEVICE_BOUNDS: return "a kernel read an index out of range (device status)";
        case MOE_ERR_ALIGN: return "a device pointer is not 16-byte aligned";
        default: return "unknown status";
    }
}

const char* moe_version(void) { return "0.1.0"; }

int moe_plan_describe(const moe_config* cfg, char* buf, size_t len) {
    MOE_TRY(check_config(cfg));
    if (!buf || len == 0) return MOE_ERR_NULL;
    const moe_config& c = *cfg;
    const char* router = use_split_d_router(c.T, c.E) ? "split_d"
                         : use_warp_router(c.E, c.d, c.dtype) ? "warp"
                                                              : "gemm";
    if (fused_decode_plan(c, false, kNominalSms).ok) {
        snprintf(buf, len, "routing=token_choice router=fused up=fused ksplit_up=1 down=fused ksplit_down=1 "
                           "gather_a=0 h=bf16");
        return MOE_OK;
    }
    const char* gemm = c.dtype != MOE_BF16 ? "simt" : (use_decode_gemm(c) ? (decode_tile_rows(c) == 32 ? "tc_decode32" : "tc_decode64") : "tc");
    const Splits sp = choose_splits(c);
    const bool gather = use_gather_a(c);
    const bool pair_up = use_pair_gemm(c) && sp.up == 1 && !gather;
    const bool pair_dn = use_pair_gemm(c) && sp.down == 1;
    snprintf(buf, len, "routing=%s router=%s up=%s%s ksplit_up=%d down=%s%s ksplit_down=%d gather_a=%d h=%s",
             expert_choice(c) ? "expert_choice" : "token_choice", router, gemm,
             pair_up ? "_pair" : "", sp.up, gemm, pair_dn ? "_pair" : "", sp.down, gather ? 1 : 0,
             use_h_split(c) ? "bf16_hi_lo" : (c.dtype == MOE_BF16 ? "bf16" : "f32"));
    return MOE_OK;
}

int moe_set_stage_events(void* const* events, int n) {
    if (!events) {
        g_stage_n = 0;
        return MOE_OK;
    }
    if (n < 0 || n > kStageEvents) return MOE_ERR_SHAPE;
    for (int i = 0; i < n; ++i) g_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
    g_stage_n = n;
    return MOE_OK;
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_test_stall_gemm(int on) { return g_test_stall.exchange(on != 0 ? 1 : 0, std::memory_order_relaxed); }

}  // extern "C"
